"""The step replayed from CUDA graphs (repstep_step_graph) through the C ABI: every output
bit equal to the oracle's, or to the ordinary step's on twin inputs, across steps whose
hyperparameters change (the AdamW node a replay rewrites), across captures forced by new
buffers, a new clip threshold or a new decay mask, beside roots pending on the hash
stream, and on another stream."""
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


def _outs():
    return (torch.empty(1, dtype=torch.float32, device=DEV),
            torch.empty(1, dtype=torch.int64, device=DEV))


def _check_against_oracle(ref, w, m, v, norm, root, t):
    U.assert_same_f32(w, ref["w"], f"w step {t}")
    U.assert_same_f32(m, ref["m"], f"m step {t}")
    U.assert_same_f32(v, ref["v"], f"v step {t}")
    U.assert_same_f32(norm, np.array([ref["norm"]], np.float32), f"norm step {t}")
    assert U.root_of(root) == ref["root"], f"root step {t}"


@pytest.mark.parametrize("n,R,dtype,hash_mode", [
    (3 * 4096 + 1234, 8, torch.float32, 0),
    (65536 + 7, 5, torch.bfloat16, 0),
    (4097, 4, torch.float32, 1),
    (1_500_001, 8, torch.float32, 0),      # two Merkle passes: the leaf pass has 2 blocks
])
def test_graph_steps_match_oracle(n, R, dtype, hash_mode):
    ctx = rs.Repstep(n, grad_dtype=dtype, device=DEV, hash_mode=hash_mode)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    norm, root = _outs()
    # one set of gradient buffers, refilled each step (a graph keeps its pointers)
    grads = U.gen_grads(n, R, 1, dtype)
    steps = 4
    for t in range(1, steps + 1):
        fresh = U.gen_grads(n, R, t, dtype, scale=(1.0, 3000.0)[t % 2])
        for g, f in zip(grads, fresh):
            g.copy_(f)
        ctx.step_graph(grads, w, m, v, U.hp_for(t), step=t, norm_out=norm, root_out=root)
        ctx.sync()
        ref = U.oracle_step(U.oracle_grads(grads), ow, om, ov, t, hash_mode=hash_mode)
        ow, om, ov = ref["w"], ref["m"], ref["v"]
        _check_against_oracle(ref, w, m, v, norm, root, t)
    assert ctx.graph_stats() == (1, steps - 1)
    ctx.destroy()


def _twins(n, R, dtype=torch.float32, **kw):
    """An ordinary and a graph context on identical inputs."""
    out = []
    for _ in range(2):
        ctx = rs.Repstep(n, grad_dtype=dtype, device=DEV, **kw)
        w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
        if kw.get("param_dtype") == torch.bfloat16:
            w = w.to(torch.bfloat16)
        out.append((ctx, [w, m, v]))
    return out


def _same_state(a, b, what):
    for x, y, name in zip(a, b, "wmv"):
        assert torch.equal(x.view(torch.int16 if x.dtype == torch.bfloat16 else torch.int32),
                           y.view(torch.int16 if y.dtype == torch.bfloat16 else torch.int32)), \
            f"{name} {what}"


@pytest.mark.parametrize("kw", [
    dict(param_dtype=torch.bfloat16),
    dict(subnormals=rs.SUBNORMALS_FTZ),
    dict(block_threads=256, grid_blocks=7),
    dict(hash_mode=rs.HASH_BLAKE2B, param_dtype=torch.bfloat16),
])
def test_graph_equals_ordinary_step_in_every_mode(kw):
    n, R = 2 * 4096 + 77, 4
    (c0, s0), (c1, s1) = _twins(n, R, **kw)
    n0, r0 = _outs()
    n1, r1 = _outs()
    grads = U.gen_grads(n, R, 1)
    for t in range(1, 5):
        for g, f in zip(grads, U.gen_grads(n, R, t, scale=(1.0, 3000.0)[t % 2])):
            g.copy_(f)
        c0.step(grads, *s0, U.hp_for(t), step=t, norm_out=n0, root_out=r0)
        c1.step_graph(grads, *s1, U.hp_for(t), step=t, norm_out=n1, root_out=r1)
        c0.sync()
        c1.sync()
        _same_state(s0, s1, f"step {t}")
        assert torch.equal(n0.view(torch.int32), n1.view(torch.int32)), f"norm step {t}"
        assert U.root_of(r0) == U.root_of(r1), f"root step {t}"
    assert c1.graph_stats() == (1, 3)


def test_graph_with_decay_mask_equals_ordinary_step():
    n, R = 3 * 4096 + 5, 4
    mask = rs.decay_mask_from_segments(n, [(0, False), (1000, True), (9000, False),
                                           (9100, True)]).to(DEV)
    (c0, s0), (c1, s1) = _twins(n, R)
    for c in (c0, c1):
        c.set_decay_mask(mask)
    n0, r0 = _outs()
    n1, r1 = _outs()
    grads = U.gen_grads(n, R, 1)
    for t in range(1, 4):
        c0.step(grads, *s0, U.hp_for(t), step=t, norm_out=n0, root_out=r0)
        c1.step_graph(grads, *s1, U.hp_for(t), step=t, norm_out=n1, root_out=r1)
        c0.sync()
        c1.sync()
        _same_state(s0, s1, f"step {t}")
        assert U.root_of(r0) == U.root_of(r1), f"root step {t}"
    # a new mask is part of what the graph is specific to
    c0.set_decay_mask(None)
    c1.set_decay_mask(None)
    c0.step(grads, *s0, U.hp_for(4), step=4, norm_out=n0, root_out=r0)
    c1.step_graph(grads, *s1, U.hp_for(4), step=4, norm_out=n1, root_out=r1)
    c0.sync()
    c1.sync()
    _same_state(s0, s1, "step 4, no mask")
    assert U.root_of(r0) == U.root_of(r1)
    assert c1.graph_stats() == (2, 2)


def test_graph_captures_again_for_new_buffers_and_clip():
    """Each change of what a graph holds forces a capture; the steps after it replay."""
    n, R = 4096 * 5 + 3, 8
    (c0, s0), (c1, s1) = _twins(n, R)
    n0, r0 = _outs()
    n1, r1 = _outs()
    grads_a = U.gen_grads(n, R, 1)
    grads_b = U.gen_grads(n, R, 2, scale=3000.0)
    plan = [  # (gradients, clip, new output tensors) per step; expected captures so far
        (grads_a, 1.0, "", 1),
        (grads_a, 1.0, "", 1),
        (grads_b, 1.0, "", 2),         # new gradient buffers
        (grads_b, 0.5, "", 3),         # new clip threshold
        (grads_b, 0.5, "norm", 4),     # a new norm output: an argument of the clip's kernel
        (grads_b, 0.5, "root", 4),     # the root passes are ordinary launches
    ]
    for t, (grads, clip, fresh_out, caps) in enumerate(plan, 1):
        if fresh_out == "norm":
            n1 = _outs()[0]
        elif fresh_out == "root":
            r1 = _outs()[1]
        c0.step(grads, *s0, U.hp_for(t, clip=clip), step=t, norm_out=n0, root_out=r0)
        c1.step_graph(grads, *s1, U.hp_for(t, clip=clip), step=t, norm_out=n1, root_out=r1)
        c0.sync()
        c1.sync()
        _same_state(s0, s1, f"step {t}")
        assert torch.equal(n0.view(torch.int32), n1.view(torch.int32)), f"norm step {t}"
        assert U.root_of(r0) == U.root_of(r1), f"root step {t}"
        assert c1.graph_stats()[0] == caps, (t, c1.graph_stats())
    # the same state arrays in a new order: the graph must not be reused
    w, m, v = s1
    c1.step_graph(grads_b, w, v, m, U.hp_for(7, clip=0.5), step=7, norm_out=n1, root_out=r1)
    c1.sync()
    assert c1.graph_stats() == (5, 2)


def test_graph_and_ordinary_steps_interleaved_with_a_hash_stream():
    """Both kinds of step leave their root pending on the hash stream, and the next step's
    AdamW, a graph's or not, waits for it."""
    n, R = 1_000_003, 8
    ctx = rs.Repstep(n, device=DEV)
    ctx.set_hash_stream(torch.cuda.Stream(DEV))
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    norm, root = _outs()
    grads = U.gen_grads(n, R, 1)
    for t in range(1, 7):
        for g, f in zip(grads, U.gen_grads(n, R, t, scale=(1.0, 3000.0)[t % 2])):
            g.copy_(f)
        fn = ctx.step_graph if t % 3 else ctx.step
        fn(grads, w, m, v, U.hp_for(t), step=t, norm_out=norm, root_out=root)
        ctx.sync()
        ref = U.oracle_step(U.oracle_grads(grads), ow, om, ov, t)
        ow, om, ov = ref["w"], ref["m"], ref["v"]
        _check_against_oracle(ref, w, m, v, norm, root, t)
    assert ctx.graph_stats() == (1, 3)


def test_graph_on_a_side_stream_and_launch_count():
    n, R = 4096 * 3, 4
    (c0, s0), (c1, s1) = _twins(n, R)
    n0, r0 = _outs()
    n1, r1 = _outs()
    grads = U.gen_grads(n, R, 1)
    side = torch.cuda.Stream(DEV)
    side.wait_stream(torch.cuda.current_stream(DEV))
    per_step = []
    for t in range(1, 4):
        c0.step(grads, *s0, U.hp_for(t), step=t, norm_out=n0, root_out=r0)
        before = c1.launch_count()
        with torch.cuda.stream(side):
            c1.step_graph(grads, *s1, U.hp_for(t), step=t, norm_out=n1, root_out=r1)
            c1.sync()
        per_step.append(c1.launch_count() - before)
        c0.sync()
        _same_state(s0, s1, f"step {t}")
        assert U.root_of(r0) == U.root_of(r1)
    # every replay runs the kernels of one ordinary step
    b0 = c0.launch_count()
    c0.step(grads, *s0, U.hp_for(4), step=4, norm_out=n0, root_out=r0)
    assert per_step == [c0.launch_count() - b0] * 3


def test_graph_step_rejects_what_the_ordinary_step_rejects():
    n, R = 4096, 2
    ctx = rs.Repstep(n, device=DEV)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    grads = U.gen_grads(n, R, 1)
    with pytest.raises(rs.RepstepError):
        ctx.step_graph(grads, w, m, v, U.hp_for(1, clip=0.0), step=1)
    big = torch.zeros(n + 4, device=DEV)
    with pytest.raises(rs.RepstepError):
        ctx.step_graph(grads, big[1:n + 1], m, v, U.hp_for(1), step=1)   # misaligned w
    assert ctx.graph_stats() == (0, 0)
    ctx.step_graph(grads, w, m, v, U.hp_for(1), step=1)
    ctx.sync()
    assert ctx.graph_stats() == (1, 0)


def test_graph_step_on_an_empty_parameter_vector():
    """n = 0 has no AdamW node, so each call captures afresh; the root is still right."""
    ctx = rs.Repstep(0, device=DEV)
    z = torch.zeros(1, dtype=torch.float32, device=DEV)
    grads = [torch.zeros(1, dtype=torch.float32, device=DEV)] * 2
    norm, root = _outs()
    e = np.zeros(0, np.float32)
    for t in (1, 2):
        ctx.step_graph(grads, z, z.clone(), z.clone(), U.hp_for(t), step=t, norm_out=norm,
                       root_out=root)
        ctx.sync()
        assert float(norm.item()) == 0.0
        assert U.root_of(root) == O.state_hash(t, e, e, e)
    assert ctx.graph_stats() == (2, 0)
