"""The C ABI library loads and exports every function include/repstep.h declares; host-only
entry points (sizes, layout, bias corrections, status names) behave as documented.  CPU
only: no call here touches a GPU."""
import ctypes as C
import os
import re
import subprocess

import numpy as np
import pytest

from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "repstep.h")


@pytest.fixture(scope="module")
def L():
    from bitwise_reproducible_step_gb300 import build
    build.build()
    return rs.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(repstep_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(rs.EXPORTS)


def test_every_declared_symbol_is_exported(L):
    out = subprocess.run(["nm", "-D", "--defined-only", rs.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\b(repstep_[a-z_]+)\b", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_status_strings(L):
    for code in range(9):
        assert rs.strerror(code) and rs.strerror(code) != "unknown status"
    assert rs.strerror(99) == "unknown status"


def test_bias_corrections_match_oracle(L):
    for t in [1, 2, 3, 5, 10, 100, 4000]:
        got = rs.bias_corrections(np.float32(0.9), np.float32(0.999), t)
        want = O.bias_corrections(0.9, 0.999, t)
        assert np.float32(got[0]).view(np.uint32) == want[0].view(np.uint32)
        assert np.float32(got[1]).view(np.uint32) == want[1].view(np.uint32)


def test_bias_corrections_match_golden_bits(L):
    """The library's host-side bias corrections against the hand-derived bit table for
    beta1 = 0.9, beta2 = 0.999 (tests/golden/bias_corrections.txt)."""
    rows = {}
    for line in open(os.path.join(ROOT, "tests", "golden", "bias_corrections.txt")):
        parts = [x.strip() for x in line.split("|")]
        if line.startswith("#") or len(parts) != 3:
            continue
        rows[int(parts[0])] = (int(parts[1], 16), int(parts[2], 16))
    b1, b2 = np.uint32(0x3F666666).view(np.float32), np.uint32(0x3F7FBE77).view(np.float32)
    assert sorted(rows) == [1, 2, 3, 5, 10]
    for t, want in rows.items():
        got = rs.bias_corrections(b1, b2, t)
        assert tuple(int(np.float32(x).view(np.uint32)) for x in got) == want, t


def test_workspace_sizes_and_layout(L):
    for n in [0, 1, 4095, 4096, 4097, 12_800_000, 1_200_000_000, 3_000_000_000, 2 ** 32 - 1]:
        b = rs.workspace_bytes(n)
        assert b >= 4 * n + 8 * (1 + 3 * ((n + 4095) // 4096))
        cfg = rs.Config(n, 0, 0, 0, 0)
        lay = rs.Layout()
        assert L.repstep_workspace_layout(C.byref(cfg), C.byref(lay)) == 0
        offs = [lay.g, lay.chunk_sums, lay.norm_partials, lay.leaves, lay.merkle_partials,
                lay.pow_table, lay.scalars, lay.total]
        assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
        assert lay.total == b
        assert lay.chunk_sums >= 4 * n and lay.leaves - lay.norm_partials >= 4


def test_bad_configs_rejected(L):
    assert rs.workspace_bytes(2 ** 32) == 0
    cfg = rs.Config(10, 5, 0, 0, 0)
    assert L.repstep_workspace_bytes(C.byref(cfg)) == 0
    cfg = rs.Config(10, 0, 0, 300, 0)
    assert L.repstep_workspace_bytes(C.byref(cfg)) == 0
    cfg = rs.Config(10, 0, -1, 0, 0)
    assert L.repstep_workspace_bytes(C.byref(cfg)) == 0
    cfg = rs.Config(10, 0, 0, 0, 0, 2, 0)     # parameter dtype neither fp32 nor bf16
    assert L.repstep_workspace_bytes(C.byref(cfg)) == 0
    cfg = rs.Config(10, 0, 0, 0, 0, 0, 2)     # subnormal mode neither IEEE nor FTZ
    assert L.repstep_workspace_bytes(C.byref(cfg)) == 0
    cfg = rs.Config(10, 0, 0, 0, 0, 0, 1)     # software flush-to-zero: a valid mode
    assert L.repstep_workspace_bytes(C.byref(cfg)) > 0


def test_bf16_parameters_need_no_more_workspace(L):
    # w lives in the caller's buffer either way; the workspace holds g (fp32) and digests
    for n in [0, 4097, 12_800_000]:
        f32 = rs.Config(n, 1, 0, 0, 0, 0, 0)
        b16 = rs.Config(n, 1, 0, 0, 0, 1, 0)
        assert L.repstep_workspace_bytes(C.byref(b16)) == L.repstep_workspace_bytes(C.byref(f32)) > 0


def test_create_rejects_before_touching_a_device(L):
    ctx = C.c_void_p()
    cfg = rs.Config(100, 0, 0, 0, 0)
    # null workspace, misaligned workspace, too small: all host-side checks
    assert L.repstep_create(C.byref(cfg), None, 10 ** 6, None, C.byref(ctx)) == 1
    assert L.repstep_create(C.byref(cfg), C.c_void_p(0x1000 + 8), 10 ** 6, None, C.byref(ctx)) == 2
    assert L.repstep_create(C.byref(cfg), C.c_void_p(0x1000), 16, None, C.byref(ctx)) == 3
    assert not ctx.value
    # every entry point rejects a null context
    assert L.repstep_reduce(None, None, 1, 1, 1, 0, 0) == 1
    assert L.repstep_clip(None, 1.0, None, None) == 1
    assert L.repstep_sync(None, None) == 1
    hp = rs.HParams()
    assert L.repstep_step(None, None, 1, 1, 1, None, None, None, C.byref(hp), 1, None,
                          None) == 1
    assert L.repstep_step_from_host(None, None, 1, None, 0, 0, None, None, None, C.byref(hp), 1,
                                    None, None) == 1
    assert L.repstep_clip_gathered(None, None, 0, 1.0, None, None) == 1
    assert L.repstep_root_gathered(None, 1, 0, None, None) == 1


def test_image_bytes(L):
    assert rs.image_bytes(12_800_000) == 153_600_008 == O.image_bytes(12_800_000)
    assert rs.image_bytes(3_000_000_000) == 36_000_000_008


@pytest.mark.parametrize("n,segs", [
    (1, [(0, True)]), (1, [(0, False)]), (31, [(0, True), (3, False), (30, True)]),
    (32, [(0, False), (31, True)]), (33, [(0, True), (32, False)]),
    (1000, [(0, True), (5, False), (64, True), (65, False), (100, True), (999, False)]),
    (100_003, [(0, False), (4096, True), (4100, False), (9000, True), (70_001, False)]),
])
def test_decay_mask_from_segments_brute_force(L, n, segs):
    got = rs.decay_mask_from_segments(n, segs).numpy().view(np.uint32)
    assert got.size == (n + 31) // 32
    want = np.zeros(got.size, np.uint32)
    for k, (b, d) in enumerate(segs):
        e = segs[k + 1][0] if k + 1 < len(segs) else n
        for i in range(b, e):
            if d:
                want[i // 32] |= np.uint32(1 << (i % 32))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("segs", [[(1, True)], [(0, True), (0, False)], [(0, True), (9, False), (7, True)],
                                  [(0, True), (100, False)], []])
def test_decay_mask_bad_segments_rejected(L, segs):
    with pytest.raises(rs.RepstepError) as ei:
        rs.decay_mask_from_segments(100, segs)
    assert ei.value.code == 1
    assert rs.decay_mask_from_segments(0, []).numel() == 0
