"""The allocation-free reduce + norm entry point (repstep_reduce_norm_noalloc).

It exists for callers that may not allocate device memory when they need the averaged
gradient and its pre-clip norm (an audit process next to a training job that owns almost
all device memory, an out-of-memory error path), so it keeps its scratch in a fixed array
inside the library.  These tests call it through the C ABI twice in a row -- with
different sizes, dtypes and data, so leftovers from an earlier call would show -- and
require the same bits as the workspace-based repstep_reduce + repstep_clip and as the
oracle, and check that a call leaves the device's free memory unchanged.  This file is
collected last on purpose; it also passes when run alone in a fresh process.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def via_workspace(grads, n, clip):
    ctx = rs.Repstep(n, grad_dtype=grads[0].dtype)
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    scale = torch.empty(1, dtype=torch.float32, device="cuda")
    ctx.reduce(grads)
    ctx.clip(clip, norm_out=norm, scale_out=scale)
    ctx.sync()
    return ctx.g_view().clone(), norm, scale


def via_noalloc(grads, n, clip):
    g = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    norm = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    scale = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    arr = (C.c_void_p * len(grads))(*[t.data_ptr() for t in grads])
    code = rs.REPSTEP_BF16 if grads[0].dtype == torch.bfloat16 else rs.REPSTEP_F32
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = rs.lib().repstep_reduce_norm_noalloc(arr, len(grads), code, n, clip,
                                              C.c_void_p(g.data_ptr()),
                                              C.c_void_p(norm.data_ptr()),
                                              C.c_void_p(scale.data_ptr()), stream)
    assert rc == 0, rs.strerror(rc)
    torch.cuda.synchronize()
    return g, norm, scale


def test_noalloc_equals_workspace_path_and_oracle_on_calls_in_a_row():
    """Three calls in a row, each against the workspace path bit for bit and against the
    oracle.  The second has n = 2^24 + 4099, so c = 4098 chunk sums take the two-pass norm
    (partials in the fixed array); the third is smaller again and in bf16, so anything the
    earlier calls left in the array would show."""
    cases = [
        (300_001, 8, torch.float32, 3000.0, 1.0),        # clipped, several norm chunks
        ((1 << 24) + 4099, 4, torch.float32, 1.0, 1.0),  # two-pass norm
        (70_003, 4, torch.bfloat16, 1.0, 0.5),           # smaller: earlier scratch left over
    ]
    for call, (n, R, dt, scale_by, clip) in enumerate(cases, 1):
        grads = U.gen_grads(n, R, 10 + call, dt, scale=scale_by)
        g_ref, n_ref, s_ref = via_workspace(grads, n, clip)
        g_got, n_got, s_got = via_noalloc(grads, n, clip)
        U.assert_same_f32(g_got, g_ref.cpu().numpy(), f"g, call {call}")
        U.assert_same_f32(n_got, n_ref.cpu().numpy(), f"norm, call {call}")
        U.assert_same_f32(s_got, s_ref.cpu().numpy(), f"scale, call {call}")
        assert np.isfinite(n_got.item()) and n_got.item() > 0
        g_o = O.reduce(U.oracle_grads(grads))
        norm_o = O.norm(g_o)
        U.assert_same_f32(g_got, g_o, f"g vs oracle, call {call}")
        U.assert_same_f32(n_got, np.array([norm_o], np.float32), f"norm vs oracle, call {call}")
        U.assert_same_f32(s_got, np.array([O.clip_scale(norm_o, clip)], np.float32),
                          f"scale vs oracle, call {call}")


def test_noalloc_call_leaves_free_device_memory_unchanged():
    """The defining property: after one call on the device (which loads the device code and
    looks up the array), further calls change the device's free memory by nothing."""
    n, R = (1 << 24) + 4099, 4
    grads = U.gen_grads(n, R, 21, torch.float32)
    via_noalloc(grads, n, 1.0)                                   # start-up call
    g = torch.empty(n, dtype=torch.float32, device="cuda")
    nrm = torch.empty(1, dtype=torch.float32, device="cuda")
    sc = torch.empty(1, dtype=torch.float32, device="cuda")
    arr = (C.c_void_p * R)(*[t.data_ptr() for t in grads])
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        rc = rs.lib().repstep_reduce_norm_noalloc(arr, R, rs.REPSTEP_F32, n, 1.0,
                                                  C.c_void_p(g.data_ptr()),
                                                  C.c_void_p(nrm.data_ptr()),
                                                  C.c_void_p(sc.data_ptr()), stream)
        assert rc == 0, rs.strerror(rc)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    g = torch.zeros(16, dtype=torch.float32, device="cuda")
    nrm = torch.zeros(1, dtype=torch.float32, device="cuda")
    arr = (C.c_void_p * 1)(g.data_ptr())
    rc = rs.lib().repstep_reduce_norm_noalloc(arr, 1, rs.REPSTEP_F32, rs.NOALLOC_MAX_N + 1, 1.0,
                                              C.c_void_p(g.data_ptr()), C.c_void_p(nrm.data_ptr()),
                                              None, None)
    assert rc == 3        # REPSTEP_ERR_SIZE, nothing enqueued
