"""The state hash's leaf digests on their own (repstep_leaves): the header leaf, then the
PF61 or BLAKE2b-64 digest of every 4096-element chunk of w, m and v ("OPEN-1B: A Fully
Auditable Training Run", App. B: a hash of parameters and optimizer state per step).  The
CUDA path against the oracle's leaves, bit for bit, and against the leaves the full hash
leaves behind.  Two states' leaf arrays differ exactly in the chunks where the states do."""
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


def u64(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


@pytest.mark.parametrize("hash_mode", [0, 1])
@pytest.mark.parametrize("n,pdt", [
    (0, torch.float32), (1, torch.float32), (4095, torch.float32), (4096, torch.bfloat16),
    (4097, torch.float32), (3 * 4096 + 1234, torch.bfloat16), (100_003, torch.float32),
])
def test_leaves_match_oracle(n, pdt, hash_mode):
    ctx = rs.Repstep(n, device=DEV, hash_mode=hash_mode, param_dtype=pdt)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    w = w.to(pdt)
    step = 7 + n % 5
    got = u64(ctx.leaves(step, w, m, v).clone())
    ctx.sync()
    wf = O.widen_bf16(U.bits16(w)) if pdt == torch.bfloat16 else w.cpu().numpy()
    want = O.leaves(step, wf, m.cpu().numpy(), v.cpu().numpy(), hash_mode=hash_mode)
    assert got.shape == want.shape == (1 + 3 * ((n + 4095) // 4096),)
    assert np.array_equal(got, want.astype(np.uint64))
    # the full hash computes the same leaves, and its root is the Merkle root over them
    root = torch.zeros(1, dtype=torch.int64, device=DEV)
    ctx.hash(step, w, m, v, root_out=root)
    ctx.sync()
    assert np.array_equal(u64(ctx.leaves_view()), got)
    assert U.root_of(root) == O.merkle_root([int(x) for x in got])


@pytest.mark.parametrize("hash_mode", [0, 1])
def test_leaves_locate_a_changed_chunk(hash_mode):
    n = 5 * 4096 + 77
    c = (n + 4095) // 4096
    ctx = rs.Repstep(n, device=DEV, hash_mode=hash_mode)
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    a = u64(ctx.leaves(3, w, m, v).clone())
    v2 = v.clone()
    e = 2 * 4096 + 11                      # chunk 2 of v
    v2[e] = torch.nextafter(v2[e], torch.tensor(float("inf"), device=DEV))
    b = u64(ctx.leaves(3, w, m, v2).clone())
    ctx.sync()
    diff = np.nonzero(a != b)[0].tolist()
    assert diff == [1 + 2 * c + 2]
    # and the header leaf follows the step
    d = u64(ctx.leaves(4, w, m, v).clone())
    ctx.sync()
    assert np.nonzero(a != d)[0].tolist() == [0]


def test_leaves_after_a_pipelined_root():
    """A leaves call waits for root passes still running on the hash stream."""
    n, R = 4 * 4096 + 9, 4
    ctx = rs.Repstep(n, device=DEV, hash_mode=rs.HASH_BLAKE2B)
    ctx.set_hash_stream(torch.cuda.Stream(DEV))
    w, m, v = I.gen_state(U.F32_WL, n=n, device=DEV)
    root = torch.zeros(1, dtype=torch.int64, device=DEV)
    ctx.step(U.gen_grads(n, R, 1), w, m, v, U.hp_for(1), step=1, root_out=root)
    got = u64(ctx.leaves(1, w, m, v).clone())
    ctx.sync()
    want = O.leaves(1, w.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy(), hash_mode=1)
    assert np.array_equal(got, want.astype(np.uint64))
    assert U.root_of(root) == O.merkle_root([int(x) for x in want])
