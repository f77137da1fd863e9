"""Checkpoint files and resume ("grow_a_language_model_checkpoints": step_NNNNNN.bin,
8 + 12n bytes) and the spike protocol (OPEN-1B §3.4.2), on the GPU against the oracle."""
import os

import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import policy as P
from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def test_checkpoint_file_bytes_and_guards(tmp_path):
    n = 3 * 4096 + 99
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    m.normal_(); v.uniform_()
    path = str(tmp_path / rs.checkpoint_name(42))
    ctx.save_checkpoint(path, 42, w, m, v)
    data = open(path, "rb").read()
    assert len(data) == 8 + 12 * n
    assert data == O.image(42, w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy())
    assert not os.path.exists(path + ".tmp")
    w2, m2, v2 = (torch.full_like(t, 7.0) for t in (w, m, v))
    assert ctx.load_checkpoint(path, w2, m2, v2) == 42
    for a, b in ((w, w2), (m, m2), (v, v2)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    # truncated, oversized and mismatched files are rejected before anything is copied
    bad = str(tmp_path / "bad.bin")
    for blob in (data[:-4096], data + b"\0\0\0\0", data[:4] + (n + 1).to_bytes(4, "little") + data[8:]):
        open(bad, "wb").write(blob)
        w3 = torch.full_like(w, 7.0)
        with pytest.raises(rs.RepstepError) as ei:
            ctx.load_checkpoint(bad, w3, m2, v2)
        assert ei.value.code == 8
        assert torch.all(w3 == 7.0)
    with pytest.raises(rs.RepstepError):
        ctx.load_checkpoint(str(tmp_path / "missing.bin"), w2, m2, v2)


def test_resume_from_checkpoint_is_bit_exact(tmp_path):
    """Save after step 2, load in a fresh context, continue: the same bits as the run that
    never stopped (the point of saving m and v on the checkpoint page)."""
    n, R, T = 5 * 4096 + 17, 4, 5
    dev = torch.device("cuda", 0)
    grads = {t: U.gen_grads(n, R, t, scale=2000.0 if t == 3 else 1.0) for t in range(1, T + 1)}
    a = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    roots_a = []
    r = torch.empty(1, dtype=torch.int64, device=dev)
    path = str(tmp_path / rs.checkpoint_name(2))
    for t in range(1, T + 1):
        a.step(grads[t], w, m, v, U.hp_for(t), step=t, root_out=r)
        a.sync()
        roots_a.append(U.root_of(r))
        if t == 2:
            a.save_checkpoint(path, t, w, m, v)
    b = rs.Repstep(n, device=dev)
    w2, m2, v2 = (torch.empty_like(x) for x in (w, m, v))
    t0 = b.load_checkpoint(path, w2, m2, v2)
    assert t0 == 2
    for t in range(t0 + 1, T + 1):
        b.step(grads[t], w2, m2, v2, U.hp_for(t), step=t, root_out=r)
        b.sync()
        assert U.root_of(r) == roots_a[t - 1]
    for x, y in ((w, w2), (m, m2), (v, v2)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))


def test_spike_protocol_matches_oracle(tmp_path):
    """A spike (pre-clip norm > 5) at training step 3 skips steps 3..7: the state stays
    bit-identical, the hash advances its header step, and AdamW resumes with t = 3."""
    n, R = 2 * 4096 + 5, 4
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    ow, om, ov = w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
    log = P.StepLog(tmp_path / "steps.jsonl")
    stepper = P.Stepper(ctx, U.HP, log=log)
    root = torch.empty(1, dtype=torch.int64, device=dev)
    adam_t = 0
    for t in range(1, 11):
        grads = U.gen_grads(n, R, t, scale=1e6 if t == 3 else 1.0)
        out = stepper.step(grads, w, m, v, train_step=t, root_out=root)
        ctx.sync()
        g = O.reduce(U.oracle_grads(grads))
        nv = O.norm(g)
        assert np.float32(out["norm"]) == nv
        applied = (t < 3) or (t > 7)
        assert out["applied"] == applied, t
        if applied:
            adam_t += 1
            bc1, bc2 = O.bias_corrections(U.HP["beta1"], U.HP["beta2"], adam_t)
            ow, om, ov = O.adamw(ow, om, ov, g, O.clip_scale(nv, U.HP["clip"]), U.HP["lr"],
                                 U.HP["beta1"], U.HP["beta2"], U.HP["eps"], U.HP["wd"], bc1, bc2)
        assert out["adam_step"] == adam_t
        U.assert_same_f32(w, ow, f"w step {t}")
        U.assert_same_f32(v, ov, f"v step {t}")
        assert U.root_of(root) == O.state_hash(t, ow, om, ov)
    # the log holds one record per step, with the norm's bits and the root of each step
    recs = log.records()
    assert [r["train_step"] for r in recs] == list(range(1, 11))
    assert [r["applied"] for r in recs] == [t < 3 or t > 7 for t in range(1, 11)]
    assert recs[-1]["root"] == P.root_hex(U.root_of(root))
    assert all(r["norm_bits"] == P.f32_bits(r["norm"]) for r in recs)
