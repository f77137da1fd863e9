"""The AdamW kernel's branch-free square root, reciprocal and division (Newton iterations
from the hardware approximations, then Markstein's correction) against the IEEE
operations, over every float of their ranges, and the update at the edges of the range
that selects them, against the oracle."""
import numpy as np
import pytest
import torch

from bitwise_reproducible_step_gb300 import repstep as rs
from oracle import oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    U.ensure_built()
    torch.cuda.set_device(0)


def test_square_root_is_ieee_on_its_whole_range():
    lo, hi = rs.SQRT_FAST_BITS
    assert rs.selftest_fast_math(0, lo, hi - lo) == 0
    assert rs.selftest_fast_math(0, 0, 1) == 0                 # +0


def test_reciprocal_is_ieee_on_its_whole_range():
    lo, hi = rs.RCP_FAST_BITS
    assert rs.selftest_fast_math(1, lo, hi - lo) == 0


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_division_is_ieee_on_random_pairs(seed):
    assert rs.selftest_fast_math(2, 0, 1 << 16, seed) == 0    # 2^26 pairs


def test_the_self_test_sees_errors():
    # outside the range the approximations flush subnormals, so the check must fail there
    assert rs.selftest_fast_math(0, 1, 1 << 20) > 0
    assert rs.selftest_fast_math(1, 1, 1 << 20) > 0


def _adamw_case(m, v, g, eps):
    n = m.size
    rng = np.random.default_rng(n)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hp = rs.hparams(lr=3e-4, beta1=0.9, beta2=0.999, eps=eps, weight_decay=0.1, clip=1e30, t=3)
    ctx = rs.Repstep(n, device=DEV)
    W, M, V, G = (torch.from_numpy(a.copy()).to(DEV) for a in (w, m, v, g))
    ctx.reduce([G])
    ctx.clip(hp.clip)
    ctx.adamw(W, M, V, hp)
    ctx.sync()
    ow, om, ov = O.adamw(w, m, v, g, 1.0, 3e-4, 0.9, 0.999, np.float32(eps), 0.1,
                         np.float32(hp.bc1), np.float32(hp.bc2))
    U.assert_same_f32(W, ow, "w")
    U.assert_same_f32(M, om, "m")
    U.assert_same_f32(V, ov, "v")


def _log_uniform(rng, n, lo, hi):
    return np.exp2(rng.uniform(lo, hi, n)).astype(np.float32)


def test_update_at_the_edges_of_the_fast_range():
    """Chunk 0 holds moments spread over the whole fast range (every warp takes the fast
    path with extreme values); chunk 1 straddles its bounds (warps fall back); chunk 2 has
    zero moments and gradients, and chunk 3 ordinary values."""
    rng = np.random.default_rng(5)
    c = 4096
    m = np.empty(4 * c, np.float32)
    v = np.empty(4 * c, np.float32)
    g = np.zeros(4 * c, np.float32)
    m[:c] = _log_uniform(rng, c, -83.8, 39.8) * rng.choice([-1, 1], c)
    v[:c] = _log_uniform(rng, c, -99.8, 39.8)
    m[c:2 * c] = _log_uniform(rng, c, -86, 42) * rng.choice([-1, 1], c)
    v[c:2 * c] = _log_uniform(rng, c, -102, 42)
    m[2 * c:3 * c] = 0.0
    v[2 * c:3 * c] = 0.0
    m[3 * c:] = (rng.standard_normal(c) * 1e-4).astype(np.float32)
    v[3 * c:] = np.abs(rng.standard_normal(c) * 1e-8).astype(np.float32)
    g[3 * c:] = (rng.standard_normal(c) * 1e-3).astype(np.float32)
    _adamw_case(m, v, g, 1e-8)


@pytest.mark.parametrize("eps", [0.0, 2.0 ** -40, 2.0 ** -41, 2.0 ** 20, 2.0 ** 21, 1e-8])
def test_update_for_eps_inside_and_outside_the_fast_range(eps):
    rng = np.random.default_rng(6)
    n = 3 * 4096 + 5
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-8).astype(np.float32)
    v[::7] = 0.0                                   # zero v' and eps = 0: u = m'/0
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[::7] = 0.0
    _adamw_case(m, v, g, eps)
