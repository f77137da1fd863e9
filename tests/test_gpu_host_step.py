"""repstep_step_from_host: a whole step whose gradients start in host memory, through the C
ABI.  The copies are pipelined over chunk-aligned ranges and several copy streams, each
range reduced as it lands; every bit must equal repstep_step on the same gradients (and the
oracle), for fp32 and bf16 gradients, ragged sizes, 1 to 64 ranges, 1 to 8 copy streams,
pinned and pageable host memory, with and without the hash stream, over consecutive steps.
Argument errors are rejected before anything is enqueued."""
import ctypes as C

import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import inputs as I
from bitwise_reproducible_step_gb300 import repstep as rs
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


CASES = [
    # n, R, dtype, pieces, copy_streams, pinned, hash_stream
    (5 * 4096 * 3 + 77, 8, torch.float32, 5, 2, True, False),
    (5 * 4096 * 3 + 77, 8, torch.float32, 1, 1, True, True),
    (300_001, 3, torch.bfloat16, 64, 8, True, False),
    (300_001, 8, torch.float32, 7, 8, False, True),
    (4096 * 64, 4, torch.float32, 64, 4, True, True),
    (1000, 2, torch.bfloat16, 0, 0, True, False),
]


@pytest.mark.parametrize("n,R,dt,pieces,cs,pinned,hstream", CASES)
def test_step_from_host_equals_step(n, R, dt, pieces, cs, pinned, hstream):
    dev = torch.device("cuda", 0)
    a, b = rs.Repstep(n, grad_dtype=dt, device=dev), rs.Repstep(n, grad_dtype=dt, device=dev)
    if hstream:
        hs = torch.cuda.Stream(dev)
        a.set_hash_stream(hs)
        b.set_hash_stream(torch.cuda.Stream(dev))
    wa, ma, va = I.gen_state(U.F32_WL, n=n, device=dev)
    wb, mb, vb = wa.clone(), ma.clone(), va.clone()
    staging = [torch.full((n,), float("nan"), dtype=dt, device=dev) for _ in range(R)]
    r = torch.empty(1, dtype=torch.int64, device=dev)
    nrm = torch.empty(1, dtype=torch.float32, device=dev)
    w_o, m_o, v_o = (x.cpu().numpy() for x in (wa, ma, va))
    for t in (1, 2, 3):
        grads = U.gen_grads(n, R, t, dt, scale=1000.0 if t == 2 else 1.0)
        host = [g.cpu() for g in grads]
        if pinned:
            host = [h.pin_memory() for h in host]
        hp = U.hp_for(t)
        a.step(grads, wa, ma, va, hp, step=t, norm_out=nrm, root_out=r)
        a.sync()
        norm_b, root_b = b.step_from_host(host, staging, wb, mb, vb, hp, step=t, pieces=pieces,
                                          copy_streams=cs)
        assert b.sync() & ~rs.FLAG_NONFINITE_NORM == 0
        U.assert_same_f32(wb, wa.cpu().numpy(), "w")
        U.assert_same_f32(mb, ma.cpu().numpy(), "m")
        U.assert_same_f32(vb, va.cpu().numpy(), "v")
        assert np.float32(norm_b).view(np.uint32) == np.float32(nrm.item()).view(np.uint32)
        assert root_b == U.root_of(r)
        o = U.oracle_step(U.oracle_grads(grads), w_o, m_o, v_o, t)
        w_o, m_o, v_o = o["w"], o["m"], o["v"]
        U.assert_same_f32(wb, w_o, "w vs oracle")
        assert np.float32(norm_b) == o["norm"] and root_b == o["root"]


def test_step_from_host_rejects_bad_arguments():
    n, R = 8192, 2
    dev = torch.device("cuda", 0)
    ctx = rs.Repstep(n, device=dev)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=dev)
    staging = [torch.zeros(n, device=dev) for _ in range(R)]
    host = [torch.zeros(n).pin_memory() for _ in range(R)]
    hp = U.hp_for(1)
    L = rs.lib()
    harr = (C.c_void_p * R)(*[h.data_ptr() for h in host])
    sarr = (C.c_void_p * R)(*[s.data_ptr() for s in staging])
    before = w.clone()

    def call(h=harr, s=sarr, R_=R, pieces=4, cs=2, wp=w.data_ptr()):
        return L.repstep_step_from_host(ctx._ctx, h, R_, s, pieces, cs, C.c_void_p(wp),
                                        C.c_void_p(m.data_ptr()), C.c_void_p(v.data_ptr()),
                                        C.byref(hp), 1, None, None)
    assert call(pieces=65) == 1                     # REPSTEP_ERR_ARG
    assert call(cs=9) == 1
    assert call(R_=0) == 1
    assert call(R_=257) == 3                        # REPSTEP_ERR_SIZE
    bad = (C.c_void_p * R)(staging[0].data_ptr() + 4, staging[1].data_ptr())
    assert call(s=bad) == 2                         # REPSTEP_ERR_ALIGN
    nul = (C.c_void_p * R)(host[0].data_ptr(), None)
    assert call(h=nul) == 1
    assert call(wp=w.data_ptr() + 4) == 2
    torch.cuda.synchronize()
    assert torch.equal(w, before)                   # nothing ran
