"""Pins for the CPU oracle: every oracle function checked against something other than
itself -- hand-derived golden values, exact rationals, closed forms, invariants, Python's
hashlib and bigint arithmetic, and torch's float64 AdamW.  CPU only.
"""
import hashlib
import math
import os
import random
import re
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests import exact as X

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
P61 = (1 << 61) - 1


def f32(x):
    return np.float32(x)


def rand_f32(rng, size, lo_exp=-30, hi_exp=10):
    """Random fp32 with random signs and exponents spread over [2^lo_exp, 2^hi_exp)."""
    mant = rng.random(size) + 1.0
    ex = rng.integers(lo_exp, hi_exp, size)
    sign = rng.choice([-1.0, 1.0], size)
    return (sign * mant * np.exp2(ex)).astype(np.float32)


# ----------------------------------------------------------------------------------
# Arithmetic model
# ----------------------------------------------------------------------------------
def test_no_contraction():
    # (1 + 2^-12)^2 = 1 + 2^-11 + 2^-24 rounds (tie to even) to 1 + 2^-11; adding
    # -(1 + 2^-11) gives 0 unfused, 2^-24 if fused into one rounding.
    a = 1.0 + 2.0 ** -12
    c = -(1.0 + 2.0 ** -11)
    assert O.probe_mul_add(a, a, c) == 0.0


def test_subnormals_kept():
    assert O.probe_subnormals()


def test_pairwise_add_is_correctly_rounded():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rand_f32(rng, 400, -149, 120), rand_f32(rng, 200, -140, -120)])
    for i in range(0, len(xs) - 1, 2):
        a, b = xs[i], xs[i + 1]
        assert X.bits(O.tree_sum(np.array([a, b], np.float32))) == X.bits(X.add(a, b))


# ----------------------------------------------------------------------------------
# Canonical tree (shape)
# ----------------------------------------------------------------------------------
def test_tree_shapes_match_golden():
    shapes = X.load_shapes(os.path.join(GOLDEN, "tree_shapes.txt"))
    rng = np.random.default_rng(2)
    for L, expr in shapes.items():
        for trial in range(40):
            x = rand_f32(rng, L, -26, 2)
            want = X.eval_shape(expr, list(x), X.add)
            got = O.tree_sum(x)
            assert X.bits(got) == X.bits(want), (L, expr, x)


def test_tree_shape_is_not_a_left_fold():
    # negative control: the golden shapes really are distinguishable from a left fold
    rng = np.random.default_rng(3)
    differs = 0
    for trial in range(200):
        x = rand_f32(rng, 7, -26, 2)
        left = x[0]
        for v in x[1:]:
            left = X.add(left, v)
        differs += X.bits(O.tree_sum(x)) != X.bits(left)
    assert differs > 0


def treefold(parts, combine):
    """Push-based binary-carry fold of the Open-1B paper, App. A.1 (Algorithm 2),
    with Result folding the leftover blocks largest-first, lower replica on the left."""
    stack = []
    for p in parts:
        level = 0
        while stack and stack[-1][0] == level:
            _, lower = stack.pop()
            p = combine(lower, p)
            level += 1
        stack.append((level, p))
    acc = stack[0][1]
    for _, p in stack[1:]:
        acc = combine(acc, p)
    return acc


@pytest.mark.parametrize("L", [1, 2, 3, 4, 5, 6, 8, 9, 10, 12, 16, 17, 20, 24, 32, 33, 48, 64])
def test_tree_equals_treefold_when_at_most_two_set_bits(L):
    assert bin(L).count("1") <= 2
    rng = np.random.default_rng(L)
    for trial in range(20):
        x = rand_f32(rng, L, -26, 2)
        assert X.bits(O.tree_sum(x)) == X.bits(treefold(list(x), X.add))


def test_tree_reading_differs_from_treefold_at_seven():
    # documented reading: with three set bits the recursive split groups the
    # remainder (4,5,6) together; the TreeFold left fold does not.
    x = np.array([1, 0, 0, 0, 2.0 ** -24, 0, 2.0 ** -24], np.float32)
    assert float(O.tree_sum(x)) == 1 + 2.0 ** -23
    assert float(treefold(list(x), X.add)) == 1.0


def _rounding_cases():
    cases = {}
    for line in open(os.path.join(GOLDEN, "rounding_cases.txt")):
        if not line.strip() or line.startswith("#") or line.startswith(("alg1_", "acc_")):
            continue
        name, ins, want, _why = [s.strip() for s in line.split("|")]
        cases[name] = (ins, X.parse_exact(want))
    return cases


def test_golden_replica_sums():
    cases = _rounding_cases()
    for name in ["sum3", "sum3b", "sum5", "sum7"]:
        ins, want = cases[name]
        vals = [float(X.parse_exact(t)) for t in ins.split(",")]
        R = len(vals)
        grads = [np.full(3, v, np.float32) for v in vals]
        g = O.reduce(grads)
        rho = X.f32(Fraction(1, R))
        expect = X.mul(np.float32(float(want)), rho)
        assert all(X.bits(x) == X.bits(expect) for x in g), (name, g, expect)


def test_golden_alg1_reductions():
    for line in open(os.path.join(GOLDEN, "rounding_cases.txt")):
        if not line.startswith("alg1_"):
            continue
        name, dps, ins, want, _why = [x.strip() for x in line.split("|")]
        dp_shard = int(dps)
        vals = [float(X.parse_exact(t)) for t in ins.split(",")]
        R = len(vals)
        g = O.reduce_alg1([np.full(3, v, np.float32) for v in vals], dp_shard)
        rho_rep = X.f32(Fraction(1, R // dp_shard))
        expect = X.mul(np.float32(float(X.parse_exact(want))), rho_rep)
        assert all(X.bits(x) == X.bits(expect) for x in g), (name, g, expect)


def test_golden_microbatch_accumulation():
    seen = 0
    for line in open(os.path.join(GOLDEN, "rounding_cases.txt")):
        if not line.startswith("acc_"):
            continue
        name, dps, acc, ins, want, _why = [x.strip() for x in line.split("|")]
        vals = [float(X.parse_exact(t)) for t in ins.split(",")]
        g = O.reduce_alg1_accum([np.full(3, v, np.float32) for v in vals], int(dps), int(acc))
        expect = np.float32(float(X.parse_exact(want)))
        assert all(X.bits(x) == X.bits(expect) for x in g), (name, g, expect)
        seen += 1
    assert seen >= 1


def test_accumulation_starts_from_positive_zero():
    # g_r <- 0 then g_r + x*rho: microbatches that are all -0 give +0 (IEEE: +0 + -0 = +0);
    # starting from the first term instead would keep -0
    mz = np.full(5, -0.0, np.float32)
    for acc in (1, 2, 3):
        g = O.reduce_alg1_accum([mz] * acc, 1, acc)
        assert np.all(g.view(np.uint32) == 0)


def test_accumulation_exact_mean_for_dyadic_inputs():
    # small integers times 2^-10 with power-of-two accum, dp_shard and dp_replicate: every
    # partial sum and every reciprocal multiply is exact, so g is the exact mean
    rng = np.random.default_rng(60)
    for rep, dps, acc in [(2, 2, 2), (4, 1, 4), (1, 4, 8), (2, 4, 2)]:
        N = rep * dps * acc
        G = [(rng.integers(-500, 500, 300) * 2.0 ** -10).astype(np.float32) for _ in range(N)]
        g = O.reduce_alg1_accum(G, dps, acc)
        for i in range(0, 300, 17):
            mean = sum(Fraction(float(x[i])) for x in G) / N
            assert Fraction(float(g[i])) == mean


def test_accumulation_with_one_microbatch_is_the_rank_gradient():
    rng = np.random.default_rng(61)
    G = [rand_f32(rng, 700, -26, 2) for _ in range(12)]
    for x in G:
        x[x == 0] = 1.0                         # no signed zeros: then 0 + x*1 = x exactly
    for dps in (1, 3, 4, 12):
        assert np.array_equal(O.reduce_alg1_accum(G, dps, 1).view(np.uint32),
                              O.reduce_alg1(G, dps).view(np.uint32))


@pytest.mark.parametrize("R", [1, 2, 4, 8, 16, 32])
def test_alg1_one_shard_power_of_two_equals_canonical_tree(R):
    # dp_shard = 1 and a power-of-two replica count: TreeFold is the perfect tree
    rng = np.random.default_rng(200 + R)
    G = [rand_f32(rng, 500, -26, 2) for _ in range(R)]
    assert np.array_equal(O.reduce_alg1(G, 1).view(np.uint32), O.reduce(G).view(np.uint32))


def test_alg1_within_error_bound_and_order_sensitive():
    rng = np.random.default_rng(31)
    for R, dps in [(6, 2), (12, 4), (12, 3), (9, 9), (10, 5)]:
        G = [(rng.standard_normal(3000) * 1e-3).astype(np.float32) for _ in range(R)]
        g = O.reduce_alg1(G, dps).astype(np.float64)
        S = np.sum([x.astype(np.float64) for x in G], axis=0)
        A = np.sum([np.abs(x.astype(np.float64)) for x in G], axis=0)
        u = 2.0 ** -24
        bound = (R + 3) * u * A / R * 1.0001 + 1e-45
        assert np.all(np.abs(g - S / R) <= bound)
    G = [rand_f32(rng, 4000, -26, 2) for _ in range(12)]
    assert not np.array_equal(O.reduce_alg1(G, 4), O.reduce_alg1(G, 3))


def test_golden_chunk_sum():
    ins, want = _rounding_cases()["chunk4096"]
    g = np.zeros(4096, np.float32)
    g[0] = 1.0
    g[2048] = 2.0 ** -12
    g[2049] = 2.0 ** -12
    _, chunks = O.norm(g, with_chunks=True)
    assert Fraction(float(chunks[0])) == want


# ----------------------------------------------------------------------------------
# Replica reduce
# ----------------------------------------------------------------------------------
def test_reduce_single_replica_is_identity():
    rng = np.random.default_rng(4)
    x = rand_f32(rng, 1000, -149, 127)
    assert np.array_equal(O.reduce([x]).view(np.uint32), x.view(np.uint32))


def test_reduce_bf16_widening_matches_torch():
    rng = np.random.default_rng(5)
    xb = torch.from_numpy(rand_f32(rng, 2000, -130, 120)).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    g = O.reduce([bits])
    assert np.array_equal(g.view(np.uint32), xb.float().numpy().view(np.uint32))


@pytest.mark.parametrize("R", [2, 4, 8, 16, 32])
def test_reduce_exact_integers(R):
    # all partial sums of small integers are exact; 1/R is exact for power-of-two R
    rng = np.random.default_rng(R)
    G = [rng.integers(-2 ** 18, 2 ** 18, 500).astype(np.float32) for _ in range(R)]
    g = O.reduce(G)
    for i in range(500):
        exact = sum(Fraction(int(G[r][i])) for r in range(R)) / R
        assert Fraction(float(g[i])) == exact


@pytest.mark.parametrize("R", [1, 2, 3, 5, 6, 7, 8, 9, 13])
def test_reduce_within_error_bound(R):
    rng = np.random.default_rng(100 + R)
    G = [(rng.standard_normal(2000) * 1e-3).astype(np.float32) for _ in range(R)]
    g = O.reduce(G).astype(np.float64)
    S = np.sum([x.astype(np.float64) for x in G], axis=0)
    A = np.sum([np.abs(x.astype(np.float64)) for x in G], axis=0)
    depth = math.ceil(math.log2(R)) if R > 1 else 0
    u = 2.0 ** -24
    bound = (depth * u * A + u * np.abs(S)) / R * 1.0001 + 1e-45
    assert np.all(np.abs(g - S / R) <= bound)


def test_reduce_replica_order_matters():
    rng = np.random.default_rng(6)
    G = [(rng.standard_normal(20000) * 10.0 ** rng.integers(-4, 4)).astype(np.float32)
         for _ in range(8)]
    a = O.reduce(G)
    b = O.reduce(G[::-1][:1] + G[1:7] + G[:1])
    assert not np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_topologies_equal_flat():
    rng = np.random.default_rng(7)
    G = [(rng.standard_normal(3000) * 1e-3).astype(np.float32) for _ in range(32)]
    flat = O.reduce(G).view(np.uint32)
    for nodes, gpn in [(1, 32), (4, 8), (8, 4), (32, 1), (2, 16), (16, 2)]:
        assert np.array_equal(O.reduce_topology(G, nodes, gpn).view(np.uint32), flat)


def test_topology_non_power_of_two_rejected():
    G = [np.zeros(4, np.float32)] * 6
    with pytest.raises(ValueError):
        O.reduce_topology(G, 2, 3)
    # one node of any size is the flat tree
    assert np.array_equal(O.reduce_topology(G, 1, 6), O.reduce(G))


# ----------------------------------------------------------------------------------
# Norm and clip
# ----------------------------------------------------------------------------------
def test_norm_single_nonzero():
    for val in [3.0, -0.75, 1e-3, 1.2345678, 2.0 ** -60]:
        for n, pos in [(1, 0), (5000, 4097), (4096, 4095), (9000, 8191)]:
            g = np.zeros(n, np.float32)
            g[pos] = val
            assert O.norm(g) == abs(np.float32(val))


@pytest.mark.parametrize("j,e", [(0, 3), (2, 10), (5, 4), (10, 7), (11, 20)])
def test_norm_constant_power_of_two(j, e):
    # g_i = 2^-e on n = 4^j elements: norm = 2^(j-e) exactly
    n = 4 ** j
    g = np.full(n, 2.0 ** -e, np.float32)
    assert float(O.norm(g)) == 2.0 ** (j - e)


def test_norm_within_error_bound():
    rng = np.random.default_rng(8)
    for n in [1, 7, 4095, 4096, 4097, 50000, 300001]:
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        exact = math.sqrt(math.fsum(float(x) * float(x) for x in g))
        c = (n + 4095) // 4096
        levels = 12 + (math.ceil(math.log2(c)) if c > 1 else 0) + 2
        assert abs(float(O.norm(g)) - exact) <= levels * 2.0 ** -24 * exact


def test_norm_tree_order_matters():
    """Negative control: the same squares summed in another order (one sequential fold
    over the whole vector, no chunks) give other bits on random data, though both stay
    within their error bounds of the exact norm.  So a bit-exact comparison of norms can
    fail, and it pins the chunked tree."""
    rng = np.random.default_rng(10)
    differing = 0
    for _ in range(8):
        g = (rng.standard_normal(3 * 4096 + 777) * 10.0 ** rng.integers(-3, 2)).astype(np.float32)
        sq = g * g                                             # fp32 products, as the method
        folded = np.sqrt(np.add.accumulate(sq, dtype=np.float32)[-1], dtype=np.float32)
        ours = O.norm(g)
        exact = math.sqrt(math.fsum(float(x) * float(x) for x in g))
        assert abs(float(ours) - exact) <= 16 * 2.0 ** -24 * exact
        assert abs(float(folded) - exact) <= g.size * 2.0 ** -24 * exact
        differing += int(np.float32(ours).view(np.uint32) != np.float32(folded).view(np.uint32))
    assert differing >= 4


def test_norm_empty_is_zero():
    assert O.norm(np.zeros(0, np.float32)) == 0.0


def test_norm_short_last_chunk_is_zero_padding():
    rng = np.random.default_rng(9)
    g = (rng.standard_normal(4096 + 1000) * 1e-2).astype(np.float32)
    padded = np.concatenate([g, np.zeros(3096, np.float32)])
    assert O.norm(g) == O.norm(padded)


def test_clip_scale():
    assert O.clip_scale(2.0, 1.0) == 0.5
    assert O.clip_scale(0.5, 1.0) == 1.0
    assert O.clip_scale(1.0, 1.0) == 1.0
    assert O.clip_scale(np.nan, 1.0) == 1.0
    assert X.bits(O.clip_scale(3.0, 1.0)) == X.bits(X.f32(Fraction(1, 3)))


# ----------------------------------------------------------------------------------
# AdamW
# ----------------------------------------------------------------------------------
B1, B2 = np.float32(0.9), np.float32(0.999)
LR, EPS, WD = np.float32(3e-4), np.float32(1e-8), np.float32(0.1)


def test_bias_corrections_step_one_and_bound():
    bc1, bc2 = O.bias_corrections(B1, B2, 1)
    assert X.bits(bc1) == X.bits(X.f32(1 - X.F(B1)))
    assert X.bits(bc2) == X.bits(X.f32(1 - X.F(B2)))
    for t in [1, 2, 3, 5, 10, 100, 1000]:
        bc1, bc2 = O.bias_corrections(B1, B2, t)
        for b, bc in [(B1, bc1), (B2, bc2)]:
            exact = 1 - float(b) ** t
            assert abs(float(bc) - exact) <= (t + 1) * 2.0 ** -24 * max(1.0, float(b) ** t) + 2 ** -24 * exact


def _golden_bits(name):
    consts, rows = {}, {}
    for line in open(os.path.join(GOLDEN, name)):
        if not line.strip() or line.startswith("#"):
            continue
        parts = [x.strip() for x in line.split("|")]
        if len(parts) == 2:
            consts[parts[0]] = int(parts[1], 16)
        else:
            rows[int(parts[0])] = (int(parts[1], 16), int(parts[2], 16))
    return consts, rows


def test_bias_corrections_match_golden_bits():
    """The t = 1, 2, 3, 5, 10 bias corrections of beta1 = 0.9 and beta2 = 0.999, bit for bit
    against the hand-derived table; the table itself re-derived here in exact rationals,
    and shown to differ from the two plausible misreadings it is meant to exclude."""
    _, rows = _golden_bits("bias_corrections.txt")
    assert sorted(rows) == [1, 2, 3, 5, 10]
    powf_differs = once_differs = 0
    for t, (want1, want2) in rows.items():
        bc1, bc2 = O.bias_corrections(B1, B2, t)
        assert (X.bits(bc1), X.bits(bc2)) == (want1, want2), t
        p1 = p2 = np.float32(1.0)
        for _ in range(t):
            p1, p2 = X.mul(p1, B1), X.mul(p2, B2)
        assert (X.bits(X.f32(1 - X.F(p1))), X.bits(X.f32(1 - X.F(p2)))) == (want1, want2)
        powf = [X.bits(X.f32(1 - X.F(X.f32(X.F(b) ** t)))) for b in (B1, B2)]
        once = [X.bits(X.f32(1 - X.F(b) ** t)) for b in (B1, B2)]
        powf_differs += powf != [want1, want2]
        once_differs += once != [want1, want2]
    assert powf_differs >= 1 and once_differs >= 1


def test_adamw_constants_match_golden_bits():
    """omega1 = 1 - beta1, omega2 = 1 - beta2 and delta = 1 - lr*wd as the oracle's AdamW
    uses them, read back through updates that expose each one alone: from m = v = 0 and
    gc = 1, m' = omega1 and v' = omega2 exactly; with g = 0, w' = w*delta."""
    consts, _ = _golden_bits("bias_corrections.txt")
    one = np.ones(1, np.float32)
    z = np.zeros(1, np.float32)
    _, m1, v1 = O.adamw(one, z, z, one, 1.0, LR, B1, B2, EPS, WD, 1.0, 1.0)
    w1, _, _ = O.adamw(one, z, z, z, 1.0, LR, B1, B2, EPS, WD, 1.0, 1.0)
    assert X.bits(m1[0]) == consts["omega1"]
    assert X.bits(v1[0]) == consts["omega2"]
    assert X.bits(w1[0]) == consts["delta"]


def _value(tok: str) -> np.float32:
    tok = tok.strip()
    sign = -1 if tok.startswith("-") else 1
    tok = tok.lstrip("-")
    if tok == "inf":
        return np.float32(sign * np.inf)
    head, *tail = re.split(r"(?<=[0-9])-(?=[0-9])", tok)     # '1-2^-20': a difference
    q = X.parse_exact(head) - sum((X.parse_exact(t) for t in tail), Fraction(0))
    assert X.F(X.f32(q)) == q, f"{tok} is not an fp32 value"
    return np.float32(sign * float(q))


def _adamw_order_cases():
    out = []
    for line in open(os.path.join(GOLDEN, "adamw_order_cases.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        name, state, hyper, want = [x.strip() for x in line.split("|")]
        out.append((name, [_value(t) for t in state.split(",")],
                    [_value(t) for t in hyper.split(",")], [_value(t) for t in want.split(",")]))
    return out


def _f32_update(w, m, v, g, scale, lr, b1, b2, eps, wd, bc1, bc2, variant=None):
    """The update in numpy fp32 scalars (each operation one IEEE rounding), with one
    misreading of the order switched in by `variant`: the negative controls."""
    f = np.float32
    with np.errstate(all="ignore"):
        om1, om2, delta = f(1) - b1, f(1) - b2, f(1) - lr * wd
        if variant == "decay_1_minus_wd":
            delta = f(1) - wd
        gc = g * scale
        m1 = b1 * m + om1 * (g if variant == "m_unclipped" else gc)
        if variant == "m_lerp":
            m1 = m + om1 * (gc - m)
        gv = g if variant == "v_unclipped" else gc
        v1 = b2 * v + om2 * (gv * gv)
        if variant == "v_omega_first":
            v1 = b2 * v + (om2 * gv) * gv
        mhat = m1 if variant == "no_bc1" else m1 / bc1
        vhat = v1 if variant == "no_bc2" else v1 / bc2
        den = np.sqrt(vhat) + eps
        if variant == "eps_in_root":
            den = np.sqrt(vhat + eps)
        elif variant == "sqrt_split":
            den = np.sqrt(v1) / np.sqrt(bc2) + eps
        u = mhat / den
        if variant == "bc1_in_denominator":
            u = m1 / (bc1 * den)
        step = lr * u
        if variant == "step_size_folded":
            step = (lr / bc1) * (m1 / den)
        w1 = w * delta - step
        if variant == "decay_after_step":
            w1 = (w - lr * u) * delta
        elif variant == "decay_in_step":
            w1 = w - lr * (u + wd * w)
    return f(w1), f(m1), f(v1)


ADAMW_VARIANTS = ["decay_1_minus_wd", "m_unclipped", "m_lerp", "v_unclipped", "v_omega_first",
                  "no_bc1", "no_bc2", "eps_in_root", "sqrt_split", "bc1_in_denominator",
                  "step_size_folded", "decay_after_step", "decay_in_step"]


def _same_bits(a, b):
    return all(X.bits(x) == X.bits(y) for x, y in zip(a, b))


def test_adamw_order_matches_golden_cases():
    """The oracle's AdamW on the hand-derived cases, every output bit equal."""
    cases = _adamw_order_cases()
    assert len(cases) == 8
    for name, (w, m, v, g, scale), (lr, b1, b2, eps, wd, bc1, bc2), want in cases:
        arr = lambda x: np.full(5, x, np.float32)  # noqa: E731
        got = O.adamw(arr(w), arr(m), arr(v), arr(g), scale, lr, b1, b2, eps, wd, bc1, bc2)
        for j in range(5):
            assert _same_bits([x[j] for x in got], want), (name, [x[j] for x in got], want)


def test_adamw_order_golden_rejects_each_misreading():
    """Negative controls: the definition restated in numpy fp32 reproduces every golden case
    (a check of the hand derivations), and each misreading of the order -- eps under the
    root, the decay after the step or inside it, the bias correction folded into the
    denominator or the step size, the square root split, the interpolation form of m, an
    unclipped gradient in either moment, a missing bias correction, delta = 1 - wd -- gives
    other bits on at least one case."""
    cases = _adamw_order_cases()
    for name, state, hyper, want in cases:
        assert _same_bits(_f32_update(*state, *hyper), want), name
    for variant in ADAMW_VARIANTS:
        caught = [name for name, state, hyper, want in cases
                  if not _same_bits(_f32_update(*state, *hyper, variant=variant), want)]
        assert caught, f"no golden case distinguishes the variant {variant}"


def test_adamw_first_step_closed_form():
    rng = np.random.default_rng(10)
    n = 3000
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    z = np.zeros(n, np.float32)
    bc1, bc2 = O.bias_corrections(B1, B2, 1)
    w1, m1, v1 = O.adamw(w, z, z, g, 1.0, LR, B1, B2, EPS, WD, bc1, bc2)
    om1 = X.f32(1 - X.F(B1))
    om2 = X.f32(1 - X.F(B2))
    for i in range(0, n, 7):
        assert X.bits(m1[i]) == X.bits(X.mul(om1, g[i])) or (g[i] == 0 and m1[i] == 0)
        assert X.bits(v1[i]) == X.bits(X.mul(om2, X.mul(g[i], g[i])))
    # |g| >> eps: the first update is lr * sign(g) up to a few ulps
    delta = float(X.f32(1 - X.F(X.mul(LR, WD))))
    g64 = g.astype(np.float64)
    approx = w.astype(np.float64) * delta - float(LR) * g64 / (np.abs(g64) + float(EPS))
    assert np.all(np.abs(w1 - approx) <= 4 * 2.0 ** -24 * (np.abs(approx) + float(LR)))


def test_adamw_no_lr_no_decay_keeps_w():
    rng = np.random.default_rng(11)
    n = 1000
    g, w = (rng.standard_normal((2, n)) * 1e-2).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-6).astype(np.float32)
    bc1, bc2 = O.bias_corrections(B1, B2, 4)
    w1, _, _ = O.adamw(w, m, v, g, 1.0, 0.0, B1, B2, EPS, 0.0, bc1, bc2)
    assert np.array_equal(w1.view(np.uint32), w.view(np.uint32))


def test_adamw_zero_gradient_only_decays():
    rng = np.random.default_rng(12)
    n = 1000
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    z = np.zeros(n, np.float32)
    bc1, bc2 = O.bias_corrections(B1, B2, 1)
    w1, m1, v1 = O.adamw(w, z, z, z, 1.0, LR, B1, B2, EPS, WD, bc1, bc2)
    delta = X.f32(1 - X.F(X.mul(LR, WD)))
    assert all(X.bits(w1[i]) == X.bits(X.mul(w[i], delta)) for i in range(n))
    assert not m1.any() and not v1.any()


def test_adamw_matches_torch_float64_over_steps():
    rng = np.random.default_rng(13)
    n, T = 4000, 6
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = [(rng.standard_normal(n) * 1e-3 * (1 + 9 * (t % 2))).astype(np.float32)
             for t in range(T)]
    # oracle
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, T + 1):
        bc1, bc2 = O.bias_corrections(B1, B2, t)
        w, m, v = O.adamw(w, m, v, grads[t - 1], 1.0, LR, B1, B2, EPS, WD, bc1, bc2)
    # torch float64 AdamW with the same fp32-valued hyperparameters
    p = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=float(LR), betas=(float(B1), float(B2)), eps=float(EPS),
                            weight_decay=float(WD), foreach=False)
    # error model: fp32 rounding (u per op) relative to the MAGNITUDES of the terms, since
    # beta1*m + (1-beta1)*g can cancel.  M bounds the m terms; the update u_t inherits
    # m's absolute error divided by the denominator, plus a few relative roundings.
    u = 2.0 ** -24
    b1, b2, lr = float(B1), float(B2), float(LR)
    M = np.zeros(n)
    tol_w = np.zeros(n)
    for t in range(1, T + 1):
        g64 = grads[t - 1].astype(np.float64)
        M = b1 * M + (1 - b1) * np.abs(g64)
        p.grad = torch.from_numpy(g64)
        opt.step()
        st = opt.state[p]
        mt, vt = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        bc1t, bc2t = 1 - b1 ** t, 1 - b2 ** t
        den = np.sqrt(vt / bc2t) + float(EPS)
        ut = (mt / bc1t) / den
        # fp32 bias corrections 1 - beta^t (repeated fp32 products) cancel: their
        # relative error is about t*u*beta^t / (1 - beta^t), large for beta2 = 0.999
        rel_bc1 = (2 * t * u * b1 ** t) / bc1t + u
        rel_bc2 = (2 * t * u * b2 ** t) / bc2t + u
        du = (4 * t * u * M / bc1t) / den + ((8 + 2 * t) * u + rel_bc1 + rel_bc2) * np.abs(ut)
        tol_w = tol_w * (1 - lr * float(WD)) + lr * du + 3 * u * (np.abs(p.detach().numpy()) + lr * np.abs(ut))
    wt = p.detach().numpy()
    st = opt.state[p]
    mt = st["exp_avg"].numpy()
    vt = st["exp_avg_sq"].numpy()
    assert np.all(np.abs(m - mt) <= 4 * T * u * M)
    assert np.all(np.abs(v - vt) <= 4 * T * u * np.abs(vt) + 1e-37)
    assert np.all(np.abs(w - wt) <= tol_w)
    # the tolerance is tight enough to catch a dropped term: skipping the decay breaks it
    w2 = w0.copy(); m2 = np.zeros(n, np.float32); v2 = np.zeros(n, np.float32)
    for t in range(1, T + 1):
        bc1, bc2 = O.bias_corrections(B1, B2, t)
        w2, m2, v2 = O.adamw(w2, m2, v2, grads[t - 1], 1.0, LR, B1, B2, EPS, 0.0, bc1, bc2)
    assert not np.all(np.abs(w2 - wt) <= tol_w)


# ----------------------------------------------------------------------------------
# PF61 leaf fingerprint
# ----------------------------------------------------------------------------------
def test_pf61_constant_definition():
    K = (math.isqrt(5 * 2 ** 122) - 2 ** 61) >> 1
    assert O.pf61_constant() == K
    assert 0 < K < P61


def test_pf61_empty_and_units():
    K = O.pf61_constant()
    assert O.pf61([]) == 0
    assert O.pf61([0]) == 1
    assert O.pf61([1]) == (1 + K) % P61
    for W in [1, 2, 5, 4096]:
        for i in sorted({0, min(1, W - 1), W // 2, W - 1}):
            x = np.zeros(W, np.uint32)
            x[i] = 1
            assert O.pf61(x) == (W + pow(K, i + 1, P61)) % P61


def test_pf61_brute_force_tiny():
    K = O.pf61_constant()
    rng = random.Random(14)
    for W in range(0, 9):
        for trial in range(30):
            x = [rng.choice([0, 1, 0xFFFFFFFF, rng.getrandbits(32)]) for _ in range(W)]
            want = (W + sum(xi * pow(K, i + 1, P61) for i, xi in enumerate(x))) % P61
            assert O.pf61(x) == want


def test_pf61_linear_and_shift():
    K = O.pf61_constant()
    rng = np.random.default_rng(15)
    for W in [3, 100, 4096]:
        x = rng.integers(0, 2 ** 31, W, dtype=np.uint64).astype(np.uint32)
        y = rng.integers(0, 2 ** 31, W, dtype=np.uint64).astype(np.uint32)
        fx, fy, fxy = O.pf61(x), O.pf61(y), O.pf61(x + y)
        assert (fxy - W) % P61 == ((fx - W) + (fy - W)) % P61
        shifted = np.concatenate([np.zeros(1, np.uint32), x])
        assert (O.pf61(shifted) - (W + 1)) % P61 == (K * (fx - W)) % P61


def test_pf61_single_word_change_always_changes_leaf():
    rng = np.random.default_rng(16)
    x = rng.integers(0, 2 ** 32, 4096, dtype=np.uint64).astype(np.uint32)
    base = O.pf61(x)
    for i in [0, 1, 2047, 4095]:
        for delta in [1, 1 << 31]:
            y = x.copy()
            y[i] ^= np.uint32(delta)
            assert O.pf61(y) != base


# ----------------------------------------------------------------------------------
# BLAKE2b nodes and the Merkle root
# ----------------------------------------------------------------------------------
@pytest.mark.parametrize("length", [0, 1, 3, 16, 64, 127, 128, 129, 255, 256, 257, 1000])
@pytest.mark.parametrize("outlen", [1, 8, 20, 32, 64])
def test_blake2b_matches_hashlib(length, outlen):
    data = bytes((i * 131 + length) & 0xFF for i in range(length))
    assert O.blake2b(data, outlen) == hashlib.blake2b(data, digest_size=outlen).digest()


def hl_node(a, b):
    d = hashlib.blake2b(a.to_bytes(8, "little") + b.to_bytes(8, "little"), digest_size=8)
    return int.from_bytes(d.digest(), "little")


def test_node_matches_hashlib():
    rng = random.Random(17)
    for _ in range(200):
        a, b = rng.getrandbits(64), rng.getrandbits(64)
        assert O.node(a, b) == hl_node(a, b)
    assert O.node(1, 2) != O.node(2, 1)


def test_merkle_shapes_match_golden():
    shapes = X.load_shapes(os.path.join(GOLDEN, "tree_shapes.txt"))
    rng = random.Random(18)
    for L, expr in shapes.items():
        leaves = [rng.getrandbits(61) for _ in range(L)]
        want = X.eval_shape(expr, leaves, hl_node)
        assert O.merkle_root(np.array(leaves, np.uint64)) == want


# ----------------------------------------------------------------------------------
# Checkpoint image and state hash
# ----------------------------------------------------------------------------------
def test_image_size_golden():
    for line in open(os.path.join(GOLDEN, "checkpoint_sizes.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        n, b, mb, mib = [int(s) for s in line.split("|")]
        assert O.image_bytes(n) == b == 8 + 12 * n
        assert round(b / 1e6) == mb
        assert math.ceil(b / 2 ** 20) == mib


def test_image_layout():
    rng = np.random.default_rng(19)
    n = 5000
    w, m, v = (rng.standard_normal((3, n))).astype(np.float32)
    img = O.image(7, w, m, v)
    assert len(img) == 8 + 12 * n
    assert int.from_bytes(img[0:4], "little") == 7
    assert int.from_bytes(img[4:8], "little") == n
    assert img[8:] == w.astype("<f4").tobytes() + m.astype("<f4").tobytes() + v.astype("<f4").tobytes()
    neg = O.image(-3, w[:1], m[:1], v[:1])
    assert int.from_bytes(neg[0:4], "little", signed=True) == -3


def test_state_hash_over_image_words():
    # leaves = header words, then 4096-word chunks of w, m, v, read from the image bytes
    rng = np.random.default_rng(20)
    for n in [0, 1, 4095, 4096, 4097, 3 * 4096 + 17]:
        w, m, v = (rng.standard_normal((3, n))).astype(np.float32)
        img = np.frombuffer(O.image(11, w, m, v), dtype="<u4")
        leaves = [O.pf61(img[0:2])]
        for a in range(3):
            arr = img[2 + a * n: 2 + (a + 1) * n]
            for k in range(0, n, 4096):
                leaves.append(O.pf61(arr[k:k + 4096]))
        assert len(leaves) == O.num_leaves(n)
        want = leaves[0] if len(leaves) == 1 else None
        root = O.state_hash(11, w, m, v)
        assert root == O.merkle_root(np.array(leaves, np.uint64))
        if want is not None:
            assert root == want


def test_state_hash_bit_flips():
    rng = np.random.default_rng(21)
    n = 3 * 4096 + 5
    w, m, v = (rng.standard_normal((3, n))).astype(np.float32)
    base = O.state_hash(1, w, m, v)
    assert O.state_hash(2, w, m, v) != base
    for arr_i in range(3):
        for pos in [0, 4096, n - 1]:
            for bit in [0, 31]:
                arrs = [w.copy(), m.copy(), v.copy()]
                arrs[arr_i].view(np.uint32)[pos] ^= np.uint32(1 << bit)
                assert O.state_hash(1, *arrs) != base


# ----------------------------------------------------------------------------------
# Whole step against torch float64 (clip + AdamW) within rounding error
# ----------------------------------------------------------------------------------
def test_step_matches_torch_float64():
    rng = np.random.default_rng(22)
    n, R, T = 9000, 4, 3
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    Gs = [[(rng.standard_normal(n) * 0.05).astype(np.float32) for _ in range(R)]
          for _ in range(T)]
    w, m, v = w0, np.zeros(n, np.float32), np.zeros(n, np.float32)
    norms = []
    for t in range(1, T + 1):
        out = O.step(Gs[t - 1], w, m, v, lr=LR, beta1=B1, beta2=B2, eps=EPS, wd=WD, clip=1.0, t=t)
        w, m, v = out["w"], out["m"], out["v"]
        norms.append(float(out["norm"]))
    assert min(norms) > 1.0  # the clip is exercised
    p = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=float(LR), betas=(float(B1), float(B2)), eps=float(EPS),
                            weight_decay=float(WD), foreach=False)
    for t in range(T):
        gm = np.mean([x.astype(np.float64) for x in Gs[t]], axis=0)
        nrm = np.sqrt(np.sum(gm * gm))
        assert abs(nrm - norms[t]) <= 1e-6 * nrm
        p.grad = torch.from_numpy(gm * min(1.0, 1.0 / nrm))
        opt.step()
    wt = p.detach().numpy()
    assert np.all(np.abs(w - wt) <= 64 * T * 2.0 ** -24 * (np.abs(wt) + float(LR)))


# ----------------------------------------------------------------------------------
# Audit-mode leaves (BLAKE2b-64 of each leaf's image bytes), pinned by hashlib
# ----------------------------------------------------------------------------------
def test_audit_leaves_match_hashlib_on_image_bytes():
    rng = np.random.default_rng(23)
    for n in [0, 1, 5, 32, 33, 4095, 4096, 4097, 2 * 4096 + 1000]:
        w, m, v = (rng.standard_normal((3, n))).astype(np.float32)
        img = O.image(9, w, m, v)
        want = [hashlib.blake2b(img[0:8], digest_size=8).digest()]
        for a in range(3):
            arr = img[8 + 4 * n * a: 8 + 4 * n * (a + 1)]
            for k in range(0, 4 * n, 4 * 4096):
                want.append(hashlib.blake2b(arr[k:k + 4 * 4096], digest_size=8).digest())
        want = [int.from_bytes(d, "little") for d in want]
        got = O.leaves(9, w, m, v, hash_mode=1)
        assert got.tolist() == want
        assert O.state_hash(9, w, m, v, hash_mode=1) == O.merkle_root(np.array(want, np.uint64))


def test_audit_and_pf61_modes_differ_but_share_the_tree():
    rng = np.random.default_rng(24)
    w, m, v = (rng.standard_normal((3, 9000))).astype(np.float32)
    assert O.state_hash(1, w, m, v, 0) != O.state_hash(1, w, m, v, 1)
    assert O.state_hash(1, w, m, v, 0) == O.merkle_root(O.leaves(1, w, m, v, 0))


# ----------------------------------------------------------------------------------
# bf16 parameters: the rounding to bf16 against torch's conversion, the update against
# the fp32 oracle on the widened value
# ----------------------------------------------------------------------------------
def test_f32_to_bf16_matches_torch_rne():
    rng = np.random.default_rng(40)
    x = np.concatenate([rand_f32(rng, 20000, -149, 127),
                        np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, 1.0039062,
                                  1.0117188, 2.0 ** -133, -(2.0 ** -149)], np.float32)])
    # ties: exactly half way between two bf16 neighbours
    ties = (rng.integers(0, 2 ** 16, 2000, dtype=np.uint64).astype(np.uint32) << 16 | 0x8000).view(np.float32)
    x = np.concatenate([x, ties[np.isfinite(ties)]]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([O.f32_to_bf16(v) for v in x], np.uint16)
    assert np.array_equal(got, want)
    assert (O.f32_to_bf16(np.float32(np.nan)) & 0x7FC0) == 0x7FC0


def test_adamw_bf16w_is_fp32_update_rounded_once():
    rng = np.random.default_rng(41)
    n = 5000
    w16 = torch.from_numpy((rng.standard_normal(n) * 0.02).astype(np.float32)).to(torch.bfloat16)
    w16 = w16.view(torch.int16).numpy().view(np.uint16)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-7).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    bc1, bc2 = O.bias_corrections(B1, B2, 3)
    w1, m1, v1 = O.adamw_bf16w(w16, m, v, g, 1.0, LR, B1, B2, EPS, WD, bc1, bc2)
    wf, mf, vf = O.adamw(O.widen_bf16(w16), m, v, g, 1.0, LR, B1, B2, EPS, WD, bc1, bc2)
    assert np.array_equal(m1.view(np.uint32), mf.view(np.uint32))
    assert np.array_equal(v1.view(np.uint32), vf.view(np.uint32))
    want = torch.from_numpy(wf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(w1, want)


# ----------------------------------------------------------------------------------
# Per-segment weight decay ("OPEN-1B", §3.2 optimizer paragraph: no decay on embeddings,
# normalisation gains or RoPE)
# ----------------------------------------------------------------------------------
SEGS = [(0, True), (5, False), (4096, True), (4100, False), (9000, True), (12_000, False)]


def _decays(n, segs):
    out = np.zeros(n, bool)
    for k, (b, d) in enumerate(segs):
        e = segs[k + 1][0] if k + 1 < len(segs) else n
        out[b:e] = d
    return out


def test_segments_zero_gradient_decays_exactly_the_decay_segments():
    # g = m = v = 0: u = 0, so a decaying element becomes w * (1 - lr wd) and any other
    # element keeps its bits -- which pins the segment lookup element by element
    n = 12_345
    rng = np.random.default_rng(50)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    z = np.zeros(n, np.float32)
    bc1, bc2 = O.bias_corrections(B1, B2, 1)
    w1, _, _ = O.adamw_segments(w, z, z, z, 1.0, LR, B1, B2, EPS, WD, bc1, bc2, SEGS)
    delta = X.f32(1 - X.F(X.mul(LR, WD)))
    dec = _decays(n, SEGS)
    want = np.where(dec, np.array([X.mul(x, delta) for x in w], np.float32), w)
    assert np.array_equal(w1.view(np.uint32), want.view(np.uint32))
    assert dec.any() and (~dec).any()


def test_segments_reduce_to_plain_adamw_per_element():
    n = 12_345
    rng = np.random.default_rng(51)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-7).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    bc1, bc2 = O.bias_corrections(B1, B2, 3)
    args = (1.0, LR, B1, B2, EPS)
    ws, ms, vs = O.adamw_segments(w, m, v, g, *args, WD, bc1, bc2, SEGS)
    wd_, md, vd = O.adamw(w, m, v, g, *args, WD, bc1, bc2)
    w0, _, _ = O.adamw(w, m, v, g, *args, 0.0, bc1, bc2)
    dec = _decays(n, SEGS)
    assert np.array_equal(ws.view(np.uint32), np.where(dec, wd_, w0).view(np.uint32))
    assert np.array_equal(ms.view(np.uint32), md.view(np.uint32))
    assert np.array_equal(vs.view(np.uint32), vd.view(np.uint32))
    # one decaying segment is plain AdamW; one non-decaying segment is AdamW with wd = 0
    assert np.array_equal(O.adamw_segments(w, m, v, g, *args, WD, bc1, bc2, [(0, 1)])[0], wd_)
    assert np.array_equal(O.adamw_segments(w, m, v, g, *args, WD, bc1, bc2, [(0, 0)])[0], w0)
    # bf16 parameters: the same choice, then one rounding
    w16 = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    b16, _, _ = O.adamw_bf16w_segments(w16, m, v, g, *args, WD, bc1, bc2, SEGS)
    d16 = O.adamw_bf16w(w16, m, v, g, *args, WD, bc1, bc2)[0]
    z16 = O.adamw_bf16w(w16, m, v, g, *args, 0.0, bc1, bc2)[0]
    assert np.array_equal(b16, np.where(dec, d16, z16))


@pytest.mark.parametrize("segs", [[(1, True)], [(0, True), (0, False)], [(0, True), (9, False), (7, True)],
                                  [(0, True), (100, False)], []])
def test_segments_bad_lists_rejected(segs):
    n = 100
    z = np.zeros(n, np.float32)
    with pytest.raises(ValueError):
        O.adamw_segments(z, z, z, z, 1.0, LR, B1, B2, EPS, WD, 1.0, 1.0, segs)


# ----------------------------------------------------------------------------------
# Software flush-to-zero mode ("OPEN-1B", §2.1 "Subnormals": FTZ zeroes subnormal
# results, DAZ subnormal inputs)
# ----------------------------------------------------------------------------------
TINY = np.float32(np.finfo(np.float32).tiny)        # 2^-126, the smallest normal


def test_flush_definition():
    rng = np.random.default_rng(70)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32)
    bits[:2000] &= 0x807FFFFF                         # plenty of subnormals and zeros
    for x in bits.view(np.float32):
        y = O.flush(x)
        if np.isnan(x):
            assert np.isnan(y)
        elif x != 0 and abs(x) < TINY:
            assert y == 0 and np.signbit(y) == np.signbit(x)
        else:
            assert X.bits(y) == X.bits(x)


def test_ftz_equals_ieee_when_nothing_is_subnormal():
    # magnitudes far from the subnormal range: every FTZ function takes exactly the IEEE
    # function's operations
    rng = np.random.default_rng(71)
    n = 9000
    G = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(6)]
    assert np.array_equal(O.reduce_ftz(G), O.reduce(G))
    assert np.array_equal(O.reduce_alg1_ftz(G, 3), O.reduce_alg1(G, 3))
    assert np.array_equal(O.reduce_alg1_ftz(G, 1, accum=2), O.reduce_alg1_accum(G, 1, 2))
    g = O.reduce(G)
    nf, cf = O.norm_ftz(g, with_chunks=True)
    ni, ci = O.norm(g, with_chunks=True)
    assert nf == ni and np.array_equal(cf, ci)
    assert O.clip_scale_ftz(np.float32(3.0), 1.0) == O.clip_scale(np.float32(3.0), 1.0)
    for t in (1, 5, 100):
        assert O.bias_corrections_ftz(B1, B2, t) == O.bias_corrections(B1, B2, t)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n) * 1e-7).astype(np.float32) + 1e-9
    bc1, bc2 = O.bias_corrections(B1, B2, 3)
    a = O.adamw_ftz(w, m, v, g, 0.5, LR, B1, B2, EPS, WD, bc1, bc2)
    b = O.adamw(w, m, v, g, 0.5, LR, B1, B2, EPS, WD, bc1, bc2)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))
    w16 = torch.from_numpy(w).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    a16 = O.adamw_ftz(w16, m, v, g, 0.5, LR, B1, B2, EPS, WD, bc1, bc2, segments=SEGS[:3])
    b16 = O.adamw_bf16w_segments(w16, m, v, g, 0.5, LR, B1, B2, EPS, WD, bc1, bc2, SEGS[:3])
    assert np.array_equal(a16[0], b16[0]) and np.array_equal(a16[1], b16[1])


def test_ftz_golden_cases():
    z = np.zeros(4, np.float32)
    # a subnormal sum is flushed: 1.5*2^-126 + (-2^-126) = 2^-127, then times 1/2
    x0, x1 = np.full(4, 1.5 * 2.0 ** -126, np.float32), np.full(4, -(2.0 ** -126), np.float32)
    assert np.all(O.reduce([x0, x1]) == np.float32(2.0 ** -128))
    g = O.reduce_ftz([x0, x1])
    assert np.all(g.view(np.uint32) == 0)                       # +0
    # DAZ on a subnormal gradient, sign kept
    g = O.reduce_ftz([np.full(4, -(2.0 ** -140), np.float32)])
    assert np.all(g.view(np.uint32) == 0x80000000)              # -0
    # tininess after rounding with an unbounded exponent: T = (3*2^22 - 1)*2^-148 times
    # fp32(1/3) = (2^25+1)/3 * 2^-25 is exactly 2^-126 - (5/12)*2^-149.  Rounded to 24
    # bits with an unbounded exponent (spacing 2^-150 below 2^-126) it is 2^-126 - 2^-150:
    # tiny, so zeroed -- although the binary32 rounding (spacing 2^-149) would give 2^-126
    T = np.full(4, float((3 * 2 ** 22 - 1) * Fraction(2) ** -148), np.float32)
    assert Fraction(float(T[0])) == (3 * 2 ** 22 - 1) * Fraction(2) ** -148
    assert np.all(O.reduce([T, z, z]) == TINY)                  # IEEE: rounds up to 2^-126
    g = O.reduce_ftz([T, z, z])
    assert np.all(g.view(np.uint32) == 0)
    # squares below the normal range vanish: a norm of 2^-70 entries is 0 in FTZ mode
    g = np.full(5000, 2.0 ** -70, np.float32)
    assert O.norm(g) > 0 and O.norm_ftz(g) == 0
    # subnormal moments are flushed: with g = 0 the update is w*(1 - lr*wd) exactly and the
    # new moments are +0 (IEEE keeps a tiny update)
    n = 6
    w = np.full(n, 0.0123, np.float32)
    m = np.full(n, 2.0 ** -130, np.float32)
    bc1, bc2 = O.bias_corrections(B1, B2, 2)
    w1, m1, v1 = O.adamw_ftz(w, m, z[:1].repeat(n), z[:1].repeat(n), 1.0, LR, B1, B2, EPS, WD,
                             bc1, bc2)
    delta = X.f32(1 - X.F(X.mul(LR, WD)))
    assert np.all(w1 == X.mul(w[0], delta))
    assert not m1.view(np.uint32).any() and not v1.view(np.uint32).any()
    wi, mi, _ = O.adamw(w, m, z[:1].repeat(n), z[:1].repeat(n), 1.0, LR, B1, B2, EPS, WD, bc1, bc2)
    assert np.all(mi != 0)


def _round24_unbounded(q: Fraction) -> Fraction:
    """q > 0 rounded to 24 significant bits, ties to even, with no exponent limit."""
    e = q.numerator.bit_length() - q.denominator.bit_length()
    while Fraction(2) ** e > q:
        e -= 1
    while Fraction(2) ** (e + 1) <= q:
        e += 1
    x = q * Fraction(2) ** (23 - e)                 # in [2^23, 2^24)
    k = x.numerator // x.denominator
    rem = x - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    return k * Fraction(2) ** (e - 23)


def _ftz_expected(exact: Fraction, ieee: np.float32) -> np.float32:
    """IEEE 754-2008 §7.5 tininess after rounding: zero the result when the exact value,
    rounded to 24 bits as though the exponent were unbounded, is nonzero and below 2^-126."""
    if exact != 0 and _round24_unbounded(abs(exact)) < Fraction(2) ** -126:
        return np.float32(-0.0) if exact < 0 else np.float32(0.0)
    return ieee


def test_ftz_tininess_is_detected_after_rounding_with_unbounded_exponent():
    one_m24 = np.float32(1 - 2.0 ** -24)            # largest float below 1
    one_m23 = np.float32(1 - 2.0 ** -23)
    one_p23_tiny = np.float32((1 + 2.0 ** -23) * 2.0 ** -126)
    # exact 2^-126 - 2^-150: representable with an unbounded exponent, so tiny; zeroed
    # with its sign although binary32 rounding gives 2^-126
    assert X.bits(O.mul_ftz(one_m24, TINY)) == 0
    assert X.bits(O.mul_ftz(-one_m24, TINY)) == 0x80000000
    assert np.float32(one_m24) * TINY == TINY
    # exact 2^-126 (1 - 2^-46): rounds (unbounded) to 2^-126, not tiny; kept.  Detecting
    # tininess before rounding would zero it
    assert O.mul_ftz(one_m23, one_p23_tiny) == TINY
    # exact 2^-126 - 2^-149: subnormal under every reading
    assert X.bits(O.mul_ftz(one_m23, TINY)) == 0
    # quotients: (1 - 2^-24) 2^-100 / 2^26 = 2^-126 - 2^-150 is tiny; 2^-100 / 2^26 is not
    assert X.bits(O.div_ftz(np.float32((1 - 2.0 ** -24) * 2.0 ** -100), 2.0 ** 26)) == 0
    assert O.div_ftz(2.0 ** -100, 2.0 ** 26) == TINY
    # DAZ: a subnormal operand is zero first
    assert X.bits(O.mul_ftz(2.0 ** -130, 2.0 ** 100)) == 0
    assert X.bits(O.div_ftz(-(2.0 ** -130), 2.0 ** -100)) == 0x80000000
    assert np.isnan(O.div_ftz(2.0 ** -130, 0.0))    # 0/0 after DAZ


def test_ftz_mul_div_against_exact_arithmetic_near_the_boundary():
    """Products and quotients built to land within a few units of 2^-126, checked
    against the rule evaluated in exact rational arithmetic."""
    rng = np.random.default_rng(72)
    for _ in range(3000):
        off = int(rng.integers(-40, 41))
        target = 2.0 ** -126 * (1 + off * 2.0 ** -26)
        # product: a in [2^-63, 2^-43), b = RN(target / a)
        a = np.float32(2.0 ** (-63 + int(rng.integers(0, 20))) * (1 + rng.random()))
        b = np.float32(target / float(a))
        with np.errstate(under="ignore"):
            ieee = np.float32(a * b)
        exact = Fraction(float(a)) * Fraction(float(b))
        assert X.bits(O.mul_ftz(a, b)) == X.bits(_ftz_expected(exact, ieee)), (a, b)
        # quotient: x in [1, 2^20), y = RN(target * x), y / x
        x = np.float32(2.0 ** int(rng.integers(0, 20)) * (1 + rng.random()))
        y = np.float32(target * float(x))
        if abs(y) < 2.0 ** -126:
            continue
        with np.errstate(under="ignore"):
            ieee = np.float32(y / x)
        exact = Fraction(float(y)) / Fraction(float(x))
        assert X.bits(O.div_ftz(y, x)) == X.bits(_ftz_expected(exact, ieee)), (y, x)
