"""Pins for the fp64 CPU oracle (no GPU).

The pages print no worked example for this path, so each oracle function is
pinned to something other than itself: closed forms, invariants, brute force
on tiny inputs, hand-derived fixtures (tests/golden/), and special cases that
reduce to an independent library routine (torch's float->bf16 rounding,
scipy's softmax, torch's scaled-dot-product attention).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
D = 128
SM = 1.0 / math.sqrt(D)


def bf16_bits(x):
    """float array -> bf16 bit patterns through torch's own RNE conversion."""
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------- bf16 rounding

@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),                  # tie between 1 and 1+2^-7 -> even (1)
    (1.0 + 3 * 2.0 ** -8, 0x3F82),              # tie between 0x3F81 and 0x3F82 -> even
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),     # just above the tie (beyond fp32 precision)
    (-2.5, 0xC020),
    (2.0 ** -133, 0x0001),                      # smallest subnormal
    (1.5 * 2.0 ** -133, 0x0002),                # subnormal tie -> even
    (2.0 ** -134, 0x0000),                      # halfway to zero -> even (zero)
    (math.ldexp(2 - 2.0 ** -8, 127), 0x7F80),   # tie above the largest finite bf16 -> even (inf)
    (math.ldexp(2 - 2.0 ** -8 - 2.0 ** -30, 127), 0x7F7F),   # just below that tie
])
def test_round_bf16_closed_forms(x, bits):
    assert oracle.round_bf16(x) == bits


def test_round_bf16_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.uniform(-30, 30, 20000),
                        rng.standard_normal(2000)]).astype(np.float32)
    ref = bf16_bits(x)
    got = np.array([oracle.round_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- summaries

def test_summary_of_identical_keys_is_the_key():
    rng = np.random.default_rng(2)
    key = bf16_bits(rng.standard_normal((5, D)))
    blocks = np.repeat(key[:, None, :], 16, axis=1)
    assert np.array_equal(oracle.summaries(blocks), key)


def test_summary_closed_form_mean():
    blocks = np.zeros((1, 16, D), np.uint16)
    blocks[0, :, 0] = bf16_bits(np.arange(16.0))         # 0..15 -> mean 7.5
    blocks[0, :, 1] = bf16_bits(np.full(16, -3.0))       # constant
    blocks[0, :8, 2] = bf16_bits(np.full(8, 1.0))        # half ones -> 0.5
    s = bits_to_f64(oracle.summaries(blocks)[0])
    assert s[0] == 7.5 and s[1] == -3.0 and s[2] == 0.5 and np.all(s[3:] == 0)


def test_summary_matches_library_mean_where_exact():
    """For N(0,1) data the fp64 sum of 16 bf16 values is exact, and where the
    mean also fits in fp32, torch's fp32->bf16 RNE gives the single rounding."""
    rng = np.random.default_rng(3)
    blocks = bf16_bits(rng.standard_normal((64, 16, D)))
    mean = bits_to_f64(blocks).mean(axis=1)               # numpy fp64 mean
    exact32 = mean.astype(np.float32).astype(np.float64) == mean
    assert exact32.mean() > 0.99
    ref = bf16_bits(mean.astype(np.float32))
    got = oracle.summaries(blocks)
    assert np.array_equal(got[exact32], ref[exact32])


# ---------------------------------------------------------------- estimator

def _unit_q(G, comps):
    q = np.zeros((G, D), np.float32)
    for h, (i, v) in enumerate(comps):
        q[h, i] = v
    return bf16_bits(q)


def test_mass_two_pages_logistic_closed_form():
    x = 1.5                                   # bf16-exact
    q = _unit_q(1, [(0, 8.0)])
    summ = np.zeros((2, D), np.float32)
    summ[0, 0] = x
    s, m = oracle.page_mass(q, bf16_bits(summ), SM)
    a = 8.0 * x * SM                          # the page-0 logit
    assert s[0, 0] == pytest.approx(a, rel=1e-15) and s[0, 1] == 0.0
    assert m[0] == pytest.approx(1.0 / (1.0 + math.exp(-a)), rel=1e-14)
    assert m[1] == pytest.approx(1.0 / (1.0 + math.exp(a)), rel=1e-14)


def test_mass_is_group_average_of_head_softmaxes():
    """Two heads that favour different pages: closed-form masses.  Taking the
    max over heads, or the softmax of the mean logit, gives other numbers."""
    x = 2.0
    q = _unit_q(2, [(0, 8.0), (1, 8.0)])
    summ = np.zeros((3, D), np.float32)
    summ[0, 0] = x
    summ[1, 1] = x
    _, m = oracle.page_mass(q, bf16_bits(summ), SM)
    ea = math.exp(8.0 * x * SM)
    assert m[0] == pytest.approx((ea + 1) / (2 * (ea + 2)), rel=1e-14)
    assert m[1] == pytest.approx((ea + 1) / (2 * (ea + 2)), rel=1e-14)
    assert m[2] == pytest.approx(1.0 / (ea + 2), rel=1e-14)


def test_mass_sums_to_one_and_single_head_is_softmax():
    rng = np.random.default_rng(4)
    q = bf16_bits(rng.standard_normal((4, D)))
    summ = bf16_bits(rng.standard_normal((300, D)) * 0.25)
    s, m = oracle.page_mass(q, summ, SM)
    assert abs(m.sum() - 1.0) < 1e-12
    assert np.all(m > 0)
    s1, m1 = oracle.page_mass(q[:1], summ, SM)
    assert np.allclose(m1, scipy.special.softmax(s1[0]), rtol=1e-12, atol=0)
    # G heads: the average of the single-head masses of each head
    avg = np.mean([oracle.page_mass(q[h:h + 1], summ, SM)[1] for h in range(4)], axis=0)
    assert np.allclose(m, avg, rtol=1e-12, atol=0)


def test_mass_invariant_to_a_common_logit_shift():
    """Adding c*e_5 to every summary adds c*q_5*sm_scale to every logit."""
    rng = np.random.default_rng(5)
    q = np.zeros((1, D), np.float32)
    q[0, :5] = [1.0, -2.0, 0.5, 3.0, 1.25]
    q[0, 5] = 4.0
    summ = np.zeros((50, D), np.float32)
    summ[:, :5] = np.round(rng.standard_normal((50, 5)) * 8) / 8     # bf16-exact
    _, m0 = oracle.page_mass(bf16_bits(q), bf16_bits(summ), SM)
    summ[:, 5] += 2.5
    _, m1 = oracle.page_mass(bf16_bits(q), bf16_bits(summ), SM)
    assert np.allclose(m0, m1, rtol=1e-12, atol=0)


# ---------------------------------------------------------------- coverage

def test_cover_golden_cases():
    with open(os.path.join(HERE, "golden", "cover_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        keep, k, _, _ = oracle.cover(np.array(c["mass"]), c["gamma"])
        assert list(np.flatnonzero(keep)) == c["kept"], c["why"]
        assert k == len(c["kept"])


def test_cover_brute_force_minimal_and_heaviest():
    """All 2^F subsets for F <= 10: the kept set has the minimal size reaching
    gamma, the largest mass among sets of that size, and the index tie-break."""
    rng = np.random.default_rng(6)
    for trial in range(150):
        F = int(rng.integers(1, 11))
        w = rng.integers(1, 9, F).astype(np.float64)          # small integers: ties happen
        mass = w / 2.0 ** math.ceil(math.log2(w.sum()))       # dyadic, total <= 1: exact sums
        # thresholds inside the range, exactly at the total, and beyond it (unreachable)
        gamma = float(rng.choice([0.3, 0.5, 0.75, 0.9, 0.99, mass.sum(), 0.999999]))
        keep, k, _, _ = oracle.cover(mass, gamma)
        best = None
        for size in range(1, F + 1):
            sets = [s for s in itertools.combinations(range(F), size) if mass[list(s)].sum() >= gamma]
            if sets:
                top = max(mass[list(s)].sum() for s in sets)
                best = (size, top, sets)
                break
        if best is None:                                      # unreachable: keep all
            assert k == F and keep.all()
            continue
        size, top, sets = best
        assert k == size
        assert mass[keep].sum() == top
        # among the heaviest minimal sets, the rule takes equal masses lower index first
        heaviest = [s for s in sets if mass[list(s)].sum() == top]
        key = lambda s: sorted(((-mass[p], p) for p in s))
        assert tuple(np.flatnonzero(keep)) == min(heaviest, key=key)


@pytest.mark.parametrize("F,gamma", [(256, 0.9), (256, 0.99), (1000, 0.4995), (8192, 0.99), (37, 0.98)])
def test_cover_uniform_gives_ceil_gamma_F(F, gamma):
    assert abs(gamma * F - round(gamma * F)) > 1e-6
    keep, k, _, _ = oracle.cover(np.full(F, 1.0 / F), gamma)
    assert k == math.ceil(gamma * F)
    assert np.array_equal(np.flatnonzero(keep), np.arange(k))   # ties -> lowest indices


def test_cover_dominant_page_and_nesting_and_gamma_one():
    rng = np.random.default_rng(7)
    F = 500
    mass = rng.random(F) * 1e-4
    mass[123] = 1.0 - mass.sum() + mass[123]
    keep, k, _, _ = oracle.cover(mass, 0.9)
    assert k == 1 and keep[123]
    mass = rng.dirichlet(np.full(F, 0.3))
    prev = np.zeros(F, bool)
    for g in [0.1, 0.3, 0.5, 0.8, 0.9, 0.95, 0.99, 0.999]:
        keep, k, _, cum = oracle.cover(mass, g)
        assert np.all(keep[prev]), "sets must nest as gamma grows"
        assert cum[k - 1] >= g and (k == 1 or cum[k - 2] < g)
        prev = keep
    keep, k, _, _ = oracle.cover(mass, 1.0)
    assert k == F and keep.all()


# ---------------------------------------------------------------- unit selection

def _pool(rng, n, Hkv=2, S=16, scale=1.0):
    return bf16_bits(rng.standard_normal((n, Hkv, S, D)) * scale)


def test_select_unit_tail_and_gamma_one():
    rng = np.random.default_rng(8)
    L = 16 * 40 + 5                                           # 40 full pages + tail
    n = 41
    kp = _pool(rng, n)
    summ = oracle.summaries(kp.reshape(-1, 16, D)).reshape(n, 2, D)
    row = rng.permutation(n).astype(np.int32)
    q = bf16_bits(rng.standard_normal((4, D)))
    lst, *_ = oracle.select_unit(q, summ, 1, row, L, 1.0, SM)
    assert list(lst) == list(range(41))
    lst, mass, *_ = oracle.select_unit(q, summ, 1, row, L, 0.5, SM)
    assert lst[-1] == 40 and np.all(np.diff(lst) > 0) and len(mass) == 40
    lst, *_ = oracle.select_unit(q, summ, 0, row, 9, 0.5, SM)   # shorter than a page
    assert list(lst) == [0]
    lst, *_ = oracle.select_unit(q, summ, 0, row, 0, 0.5, SM)   # empty context
    assert len(lst) == 0


def test_select_unit_uniform_and_dominant_and_permutation():
    rng = np.random.default_rng(9)
    F, Hkv = 200, 1
    key = bf16_bits(rng.standard_normal(D))
    summ = np.repeat(key[None, None, :], F, 0)                # identical summaries
    q = bf16_bits(rng.standard_normal((4, D)))
    row = np.arange(F, dtype=np.int32)
    lst, *_ = oracle.select_unit(q, summ, 0, row, F * 16, 0.9, SM)
    assert list(lst) == list(range(180))                     # ceil(0.9*200), lowest indices
    summ2 = bf16_bits(rng.standard_normal((F, Hkv, D)) * 0.25)
    qd = bits_to_f64(q).mean(0)
    summ2[77, 0] = bf16_bits(8.0 * qd / np.linalg.norm(qd) * math.sqrt(D))
    lst, *_ = oracle.select_unit(q, summ2, 0, row, F * 16, 0.99, SM)
    assert list(lst) == [77]
    # physical placement does not matter
    perm = rng.permutation(F).astype(np.int32)
    pool = np.empty_like(summ2)
    pool[perm] = summ2
    for g in (0.5, 0.9, 0.99):
        a, *_ = oracle.select_unit(q, summ2, 0, row, F * 16 + 3, g, SM)
        b, *_ = oracle.select_unit(q, pool, 0, perm, F * 16 + 3, g, SM)
        assert np.array_equal(a, b)


# ---------------------------------------------------------------- alternative rules

def _dominance_set(m, k):
    """Brute force: the k-subsets S where every kept page outranks every
    dropped one (larger mass, or equal mass and lower index)."""
    F = len(m)
    out = []
    for S in itertools.combinations(range(F), k):
        rest = [q for q in range(F) if q not in S]
        if all(m[p] > m[q] or (m[p] == m[q] and p < q) for p in S for q in rest):
            out.append(set(S))
    return out


def test_topk_brute_force_unique_and_heaviest():
    rng = np.random.default_rng(21)
    for trial in range(60):
        F = int(rng.integers(1, 10))
        m = rng.integers(0, 4, F).astype(np.float64)        # many ties
        m = m / m.sum() if m.sum() > 0 else np.full(F, 1.0 / F)
        for k in range(0, F + 2):
            keep = oracle.topk(m, k)
            kk = min(k, F)
            sets = _dominance_set(m, kk)
            assert len(sets) == 1                            # the order is total
            assert set(np.flatnonzero(keep)) == sets[0]
            best = max(sum(m[list(S)]) for S in itertools.combinations(range(F), kk))
            assert math.isclose(m[keep].sum(), best, abs_tol=1e-15)


def test_topk_uniform_nesting_and_limits():
    F = 37
    m = np.full(F, 1.0 / F)
    assert np.array_equal(np.flatnonzero(oracle.topk(m, 5)), np.arange(5))   # ties: lowest indices
    assert oracle.topk(m, 0).sum() == 0 and oracle.topk(m, F + 9).all()
    rng = np.random.default_rng(22)
    m = rng.dirichlet(np.full(F, 0.3))
    prev = np.zeros(F, bool)
    for k in range(F + 1):
        cur = oracle.topk(m, k)
        assert cur.sum() == k and np.all(cur >= prev)        # nested in k
        prev = cur


def test_topdelta_threshold_definition_and_relation_to_topk():
    rng = np.random.default_rng(23)
    for trial in range(40):
        F = int(rng.integers(1, 60))
        m = rng.dirichlet(np.full(F, 0.5))
        mx = m.max()
        for delta in (1.0, 0.9, 0.5, 0.1, 1e-3, 0.0, -1.0):
            keep = oracle.topdelta(m, delta)
            # restated from the definition, not from the oracle
            assert np.array_equal(keep, m >= delta * mx)
            # without ties a threshold set is a prefix of the rule order
            assert np.array_equal(keep, oracle.topk(m, int(keep.sum())))
        assert oracle.topdelta(m, 1.0).sum() == int((m == mx).sum())
        assert oracle.topdelta(m, 0.0).all()
    m = np.array([0.25, 0.25, 0.5, 0.0])
    assert list(oracle.topdelta(m, 0.5)) == [True, True, True, False]     # >= at the threshold
    assert list(oracle.topdelta(m, 0.51)) == [False, False, True, False]


def test_select_unit_rule_matches_mass_level_rules():
    rng = np.random.default_rng(24)
    n = 61
    L = 16 * 60 + 7                                          # 60 full pages + tail
    kp = _pool(rng, n)
    summ = oracle.summaries(kp.reshape(-1, 16, D)).reshape(n, 2, D)
    row = rng.permutation(n).astype(np.int32)
    q = bf16_bits(rng.standard_normal((4, D)))
    base, mass, *_ = oracle.select_unit(q, summ, 1, row, L, 0.9, SM)
    a = oracle.select_unit_rule(q, summ, 1, row, L, oracle.RULE_COVERAGE, 0.9, SM)
    assert np.array_equal(a, base)
    for k in (0, 1, 7, 60, 99):
        lst = oracle.select_unit_rule(q, summ, 1, row, L, oracle.RULE_TOPK, k, SM)
        want = list(np.flatnonzero(oracle.topk(mass, k))) + [60]
        assert list(lst) == want
    for delta in (0.9, 0.1, 1e-4):
        lst = oracle.select_unit_rule(q, summ, 1, row, L, oracle.RULE_TOPDELTA, delta, SM)
        want = list(np.flatnonzero(mass >= delta * mass.max())) + [60]
        assert list(lst) == want
    assert list(oracle.select_unit_rule(q, summ, 1, row, 9, oracle.RULE_TOPK, 3, SM)) == [0]   # tail only


# ---------------------------------------------------------------- attention

def _sdpa(q, k, v, scale):
    """torch fp64 scaled-dot-product attention, an independent implementation."""
    qt = torch.from_numpy(q)[None, :, None, :]                 # [1][G][1][d]
    kt = torch.from_numpy(k)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(v)[None, None].expand(1, q.shape[0], -1, -1)
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, :, 0].numpy()


def test_attend_dense_equals_library_attention():
    rng = np.random.default_rng(10)
    L, Hkv = 16 * 30 + 11, 2
    n = 31
    kp, vp = _pool(rng, n), _pool(rng, n)
    row = rng.permutation(n).astype(np.int32)
    q = bf16_bits(rng.standard_normal((4, D)) * 2)
    for j in range(Hkv):
        out = oracle.attend_unit(q, kp, vp, j, row, np.arange(n, dtype=np.int32), L, SM)
        kk = bits_to_f64(kp[row, j].reshape(-1, D))[:L]
        vv = bits_to_f64(vp[row, j].reshape(-1, D))[:L]
        ref = _sdpa(bits_to_f64(q), kk, vv, SM)
        assert np.allclose(out, ref, rtol=0, atol=1e-12)


def test_attend_single_token_order_convexity_and_empty():
    rng = np.random.default_rng(11)
    n = 12
    kp, vp = _pool(rng, n, Hkv=1), _pool(rng, n, Hkv=1)
    row = np.arange(n, dtype=np.int32)
    q = bf16_bits(rng.standard_normal((4, D)))
    out = oracle.attend_unit(q, kp, vp, 0, row, np.array([0], np.int32), 1, SM)
    assert np.array_equal(out, np.repeat(bits_to_f64(vp[0, 0, 0])[None], 4, 0))
    lst = np.array([1, 4, 5, 9], np.int32)
    a = oracle.attend_unit(q, kp, vp, 0, row, lst, n * 16, SM)
    b = oracle.attend_unit(q, kp, vp, 0, row, lst[::-1].copy(), n * 16, SM)
    assert np.allclose(a, b, rtol=0, atol=1e-13)
    vv = bits_to_f64(vp[lst, 0].reshape(-1, D))
    assert np.all(a <= vv.max(0) + 1e-12) and np.all(a >= vv.min(0) - 1e-12)
    z = oracle.attend_unit(q, kp, vp, 0, row, np.zeros(0, np.int32), n * 16, SM)
    assert np.all(z == 0)


def test_attend_tail_page_reads_only_valid_tokens():
    rng = np.random.default_rng(12)
    n = 3
    kp, vp = _pool(rng, n, Hkv=1), _pool(rng, n, Hkv=1)
    row = np.arange(n, dtype=np.int32)
    q = bf16_bits(rng.standard_normal((4, D)))
    L = 2 * 16 + 5
    a = oracle.attend_unit(q, kp, vp, 0, row, np.arange(3, dtype=np.int32), L, SM)
    kp2, vp2 = kp.copy(), vp.copy()
    kp2[2, 0, 5:] = bf16_bits(np.full((11, D), 1e30))         # garbage past the tail
    vp2[2, 0, 5:] = bf16_bits(np.full((11, D), -7e30))
    b = oracle.attend_unit(q, kp2, vp2, 0, row, np.arange(3, dtype=np.int32), L, SM)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- whole step

def test_decode_step_matches_units_and_library_attention():
    """The step loop's layer/request/GQA indexing: gamma=1 against torch
    attention per query head with KV head h // G, and gamma<1 against the
    per-unit functions."""
    rng = np.random.default_rng(13)
    Lyr, B, Hq, Hkv, S = 2, 3, 8, 2, 16
    seq = np.array([16 * 7 + 3, 16 * 5, 16 * 9 + 15], np.int32)
    n = [int(L) // S + (int(L) % S != 0) for L in seq]
    P = sum(n)
    perm = rng.permutation(P).astype(np.int32)
    pt = np.full((B, max(n) + 2), -1, np.int32)
    o = 0
    for r in range(B):
        pt[r, :n[r]] = perm[o:o + n[r]]
        o += n[r]
    kp = bf16_bits(rng.standard_normal((Lyr, P, Hkv, S, D)))
    vp = bf16_bits(rng.standard_normal((Lyr, P, Hkv, S, D)))
    summ = oracle.summaries(kp.reshape(-1, S, D)).reshape(Lyr, P, Hkv, D)
    q = bf16_bits(rng.standard_normal((Lyr, B, Hq, D)))
    lengths, out, used = oracle.decode_step(q, summ, kp, vp, pt, seq, 1.0, SM, n_threads=2)
    assert used >= 1
    G = Hq // Hkv
    for l in range(Lyr):
        for r in range(B):
            for h in range(Hq):
                j = h // G
                kk = bits_to_f64(kp[l, pt[r, :n[r]], j].reshape(-1, D))[:seq[r]]
                vv = bits_to_f64(vp[l, pt[r, :n[r]], j].reshape(-1, D))[:seq[r]]
                ref = _sdpa(bits_to_f64(q[l, r, h:h + 1]), kk, vv, SM)
                assert np.allclose(out[l, r, h], ref[0], rtol=0, atol=1e-12)
            assert np.all(lengths[l, r] == n[r])
    lengths, out, _ = oracle.decode_step(q, summ, kp, vp, pt, seq, 0.6, SM)
    for l in range(Lyr):
        for r in range(B):
            for j in range(Hkv):
                qg = q[l, r, j * G:(j + 1) * G]
                lst, *_ = oracle.select_unit(qg, summ[l], j, pt[r], int(seq[r]), 0.6, SM)
                assert lengths[l, r, j] == len(lst)
                ref = oracle.attend_unit(qg, kp[l], vp[l], j, pt[r], lst, int(seq[r]), SM)
                assert np.array_equal(out[l, r, j * G:(j + 1) * G], ref)
