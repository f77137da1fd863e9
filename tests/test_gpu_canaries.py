"""Out-of-bounds and unwritten-slot checks with sentinel bytes (no sanitizer runs here).

The workspace and every caller array sit inside larger buffers prefilled with a sentinel
pattern.  After steps over shard ranges with ragged edges:
- no byte outside the workspace, or outside [begin, end) of an updated range, changes;
- the alignment padding after the workspace regions of known extent still holds the
  sentinel;
- every slot the step must write (g, the chunk sums, the leaves) was overwritten."""
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
SENT = 0xA5                      # sentinel byte; 0xA5A5A5A5 as fp32 is -2.87e-16
GUARD = 64 * 1024                # guard bytes on each side (a multiple of 256)


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def guarded(nbytes: int):
    """A sentinel-filled byte buffer with the usable region [GUARD, GUARD + nbytes)."""
    buf = torch.full((GUARD + nbytes + GUARD,), SENT, dtype=torch.uint8, device=DEV)
    return buf, buf[GUARD:GUARD + nbytes]


def intact(b: torch.Tensor) -> bool:
    return bool((b == SENT).all().item())


def guards_intact(buf: torch.Tensor, nbytes: int) -> bool:
    return intact(buf[:GUARD]) and intact(buf[GUARD + nbytes:])


@pytest.mark.parametrize("hash_mode,pdt", [(0, torch.float32), (1, torch.float32),
                                           (0, torch.bfloat16)])
def test_workspace_guards_and_padding(hash_mode, pdt):
    n, R = 3 * 4096 * 7 + 1001, 5
    probe = rs.Repstep(n, device=DEV, hash_mode=hash_mode, param_dtype=pdt)
    nbytes = probe.workspace.numel()
    lay = probe.layout
    probe.destroy()
    wbuf, ws = guarded(nbytes)
    ctx = rs.Repstep(n, device=DEV, hash_mode=hash_mode, param_dtype=pdt, workspace=ws)
    c = ctx.c
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    w = w.to(pdt)
    ranges = I.shard_ranges(n, 3)
    for t in (1, 2):
        grads = U.gen_grads(n, R, t, scale=2000.0 if t == 2 else 1.0)
        for lo, hi in ranges:
            ctx.reduce(grads, begin=lo, count=hi - lo)
        ctx.clip(U.hp_for(t).clip)
        for lo, hi in ranges:
            ctx.adamw(w, m, v, U.hp_for(t), begin=lo, count=hi - lo)
        ctx.root(t)
    ctx.sync()
    assert guards_intact(wbuf, nbytes)
    # padding after the regions whose extent the layout fixes
    for off, used, nxt in ((lay.g, 4 * n, lay.chunk_sums), (lay.chunk_sums, 4 * c, lay.norm_partials),
                           (lay.leaves, 8 * (1 + 3 * c), lay.merkle_partials)):
        assert intact(ws[off + used:nxt]), f"padding after offset {off} written"
    # every slot written
    sent32 = int.from_bytes(bytes([SENT] * 4), "little", signed=True)
    sent64 = int.from_bytes(bytes([SENT] * 8), "little", signed=True)
    assert not (ctx.g_view().view(torch.int32) == sent32).any().item()
    assert not (ctx.chunk_sums_view().view(torch.int32) == sent32).any().item()
    assert not (ctx.leaves_view() == sent64).any().item()


@pytest.mark.parametrize("pdt", [torch.float32, torch.bfloat16])
def test_updates_stay_inside_their_range(pdt):
    """AdamW over [lo, hi) with ragged edges leaves every other element, and the bytes
    around the arrays, as they were."""
    n, R = 5 * 4096 + 333, 4
    es = 2 if pdt == torch.bfloat16 else 4
    ctx = rs.Repstep(n, device=DEV, param_dtype=pdt)
    bw, wb = guarded(es * n)
    bm, mb = guarded(4 * n)
    bv, vb = guarded(4 * n)
    w0, m0, v0 = I.gen_state(U.F32_WL, n=n, device=DEV)
    w = wb.view(pdt)
    w.copy_(w0.to(pdt))
    m = mb.view(torch.float32)
    m.copy_(m0)
    v = vb.view(torch.float32)
    v.copy_(v0)
    before = [t.clone() for t in (w, m, v)]
    ctx.reduce(U.gen_grads(n, R, 1))
    ctx.clip(U.hp_for(1).clip)
    lo, hi = 4096 + 3, 3 * 4096 + 4091         # both edges inside a chunk, neither 4-aligned
    ctx.adamw(w, m, v, U.hp_for(1), begin=lo, count=hi - lo)
    ctx.sync()
    for buf, nb in ((bw, es * n), (bm, 4 * n), (bv, 4 * n)):
        assert guards_intact(buf, nb)
    for now, was in zip((w, m, v), before):
        a = now.view(torch.int16 if pdt == torch.bfloat16 and now is w else torch.int32)
        b = was.view(a.dtype)
        assert torch.equal(a[:lo], b[:lo]) and torch.equal(a[hi:], b[hi:])
        assert not torch.equal(a[lo:hi], b[lo:hi])


def test_reduce_writes_only_its_range_of_g():
    n, R = 4 * 4096 + 77, 3
    probe = rs.Repstep(n, device=DEV)
    nbytes = probe.workspace.numel()
    probe.destroy()
    wbuf, ws = guarded(nbytes)
    ctx = rs.Repstep(n, device=DEV, workspace=ws)
    lo, hi = 4096 + 5, 2 * 4096 + 4093
    ctx.reduce(U.gen_grads(n, R, 1), begin=lo, count=hi - lo)
    ctx.sync()
    g = ctx.g_view().view(torch.uint8)
    assert intact(g[:4 * lo]) and intact(g[4 * hi:])
    assert guards_intact(wbuf, nbytes)


def test_caller_workspace_is_checked():
    probe = rs.Repstep(1000, device=DEV)
    nbytes = probe.workspace.numel()
    with pytest.raises(ValueError):
        rs.Repstep(1000, device=DEV, workspace=torch.empty(nbytes - 1, dtype=torch.uint8, device=DEV))
    with pytest.raises(ValueError):
        rs.Repstep(1000, device=DEV, workspace=torch.empty(nbytes, dtype=torch.float32, device=DEV))
    buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(rs.RepstepError):        # not 256-byte aligned
        rs.Repstep(1000, device=DEV, workspace=buf[16:16 + nbytes])
