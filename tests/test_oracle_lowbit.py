"""Pins for the oracle's low-bit page summaries (no GPU).

The low-bit summary is a mid-rise quantisation of the page's fp64 mean key
("Faster Flash Decoding", section 3.1: symmetric mid-rise quantiser for the
low-bit key thumbnails).  Each pin below is fixed by that definition or by
arithmetic, not by the oracle itself: summaries whose mean sits exactly on
a quantiser level, the half-step reconstruction bound, sign preservation,
the extreme codes, exact scaling laws, and agreement with the independently
pinned bf16 estimator where the two summaries stand for the same vector.
"""
import math

import numpy as np
import pytest
import torch

from oracle import oracle

D = 128
S = 16
SM = 1.0 / math.sqrt(D)


def bf16_bits(x):
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def half_levels(bits):
    return 2 ** (bits - 1)


def pages_with_mean(means):
    """Pages whose fp64 token mean is exactly `means` [n][d] (values that are
    bf16 after doubling): tokens alternate 2*mean and 0."""
    means = np.asarray(means, np.float64)
    n = means.shape[0]
    k = np.zeros((n, S, D), np.float64)
    k[:, 0::2, :] = 2.0 * means[:, None, :]
    kb = bf16_bits(k)
    assert np.array_equal(bits_to_f64(kb), k.astype(np.float32).astype(np.float64)), "not bf16-exact"
    assert np.array_equal(bits_to_f64(kb).mean(axis=1), means)
    return kb


def level_means(rng, bits, n, step):
    """Means that sit on the quantiser's levels (code + 1/2) * step, with both
    outermost levels present so that max |mean| = (2^(bits-1) - 1/2) * step."""
    h = half_levels(bits)
    codes = rng.integers(-h, h, size=(n, D))
    codes[:, 0] = h - 1
    codes[:, 1] = -h
    return codes, (codes + 0.5) * step


@pytest.mark.parametrize("bits,step", [(8, 2.0 ** -7), (8, 2.0 ** -10), (2, 0.5), (2, 2.0 ** -6)])
def test_levels_are_reproduced_exactly(bits, step):
    rng = np.random.default_rng(bits * 100 + int(-math.log2(step)))
    codes, means = level_means(rng, bits, 12, step)
    got_codes, got_steps = oracle.summaries_lowbit(pages_with_mean(means), bits)
    assert np.all(got_steps == np.float32(step))
    assert np.array_equal(got_codes.astype(np.int64), codes)


def test_codes_are_taken_against_the_stored_fp32_step():
    """a = 51 * 2^-6 and x = 2^-5: the real quotient x / (a / 127.5) is exactly
    5, but a / 127.5 = 0.4 * 2^-6 rounds UP to fp32 (0.4 -> 0x3ECCCCCD), so the
    quotient against the stored step is just below 5 and the code is 4.  Codes
    taken against the unrounded step would be 5, and (5 + 1/2) * stored step
    would then miss x by more than half a step."""
    means = np.zeros((1, D))
    means[0, 0] = 51 * 2.0 ** -6
    means[0, 1] = 2.0 ** -5
    means[0, 2] = -2.0 ** -5
    codes, steps = oracle.summaries_lowbit(pages_with_mean(means), 8)
    assert steps[0] == np.float32(0.4) * np.float32(2.0 ** -6)
    assert float(steps[0]) > 0.00625
    assert codes[0, 0] == 127 and codes[0, 1] == 4 and codes[0, 2] == -5
    assert np.all(codes[0, 3:] == 0)                     # floor(0) = 0: value +step/2


@pytest.mark.parametrize("sign", [1, -1])
def test_subnormal_step_keeps_codes_in_range(sign):
    """One token holds the smallest bf16 subnormal 2^-133, so the mean is
    a = 2^-137 and a / 127.5 = 32.125 * 2^-149 rounds to the fp32 subnormal
    32 * 2^-149 = 2^-144: the quotient a / step is 128, one past the top code,
    and the clamp holds it at 127 (at -128 for a negative mean, which is in
    range)."""
    k = np.zeros((1, S, D), np.uint16)
    k[0, 3, 9] = 0x0001 if sign > 0 else 0x8001
    codes, steps = oracle.summaries_lowbit(k, 8)
    assert float(steps[0]) == 2.0 ** -144
    assert codes[0, 9] == (127 if sign > 0 else -128)
    val = (codes[0, 9] + 0.5) * 2.0 ** -144
    assert abs(val - sign * 2.0 ** -137) <= 0.5 * 2.0 ** -144


@pytest.mark.parametrize("bits", [8, 2])
def test_half_step_bound_sign_and_extreme_codes(bits):
    rng = np.random.default_rng(7 + bits)
    q_hat = rng.standard_normal(D)
    k = rng.standard_normal((64, S, D))
    k[:16] += 3.0 * q_hat                     # planted pages (a strong shared direction)
    k[16:24] *= 1e-3                          # small magnitudes
    k[24:32] *= 1e3                           # large magnitudes
    kb = bf16_bits(k)
    mean = bits_to_f64(kb).mean(axis=1)       # the fp64 token mean of the bf16 keys
    codes, steps = oracle.summaries_lowbit(kb, bits)
    h = half_levels(bits)
    step = steps.astype(np.float64)[:, None]
    val = (codes.astype(np.float64) + 0.5) * step
    a = np.abs(mean).max(axis=1)
    # the step is a / (2^(bits-1) - 1/2) rounded once to fp32
    assert np.all(np.abs(steps.astype(np.float64) - a / (h - 0.5)) <= 2.0 ** -24 * a / (h - 0.5))
    assert codes.min() >= -h and codes.max() <= h - 1
    assert np.all(np.abs(val - mean) <= 0.5 * step * (1 + 1e-12))
    nz = mean != 0
    assert np.all(np.sign(val[nz]) == np.sign(mean[nz]))           # mid-rise: no zero level
    imax = np.abs(mean).argmax(axis=1)
    ext = codes[np.arange(len(codes)), imax].astype(np.int64)
    sgn = np.sign(mean[np.arange(len(codes)), imax])
    assert np.all(ext == np.where(sgn > 0, h - 1, -h))


def test_zero_and_non_finite_pages_give_zero_summaries():
    k = np.zeros((3, S, D), np.float32)
    k[1, 5, 7] = np.inf
    k[2, 3, 1] = np.nan
    k[2, 0, 0] = 1.0
    for bits in (8, 2):
        codes, steps = oracle.summaries_lowbit(bf16_bits(k), bits)
        assert np.all(steps == 0) and np.all(codes == 0)


@pytest.mark.parametrize("bits", [8, 2])
def test_power_of_two_scaling_and_negation(bits):
    rng = np.random.default_rng(11 + bits)
    k = bf16_bits(rng.standard_normal((24, S, D)))
    kf = bits_to_f64(k)
    c0, s0 = oracle.summaries_lowbit(k, bits)
    for f in (2.0, 0.25, 1024.0):                 # exact in bf16 and in every later step
        c1, s1 = oracle.summaries_lowbit(bf16_bits(kf * f), bits)
        assert np.array_equal(c1, c0)
        assert np.array_equal(s1.astype(np.float64), s0.astype(np.float64) * f)
    cn, sn = oracle.summaries_lowbit(bf16_bits(-kf), bits)
    assert np.array_equal(sn, s0)
    # floor(-x) = -1 - floor(x) unless x is a whole number
    mean = kf.mean(axis=1)
    x = mean / s0.astype(np.float64)[:, None]
    off_grid = x != np.floor(x)
    assert off_grid.mean() > 0.99
    assert np.array_equal(cn.astype(np.int64)[off_grid], -1 - c0.astype(np.int64)[off_grid])


def _pool_of_levels(rng, P, Hkv, bits, step):
    codes, means = level_means(rng, bits, P * Hkv, step)
    kb = pages_with_mean(means).reshape(P, Hkv, S, D)
    return codes.reshape(P, Hkv, D), means.reshape(P, Hkv, D), kb


@pytest.mark.parametrize("bits,step", [(8, 2.0 ** -7), (2, 0.5)])
def test_select_matches_bf16_estimator_when_the_summaries_coincide(bits, step):
    """Means on the quantiser's levels are bf16-exact too, so the bf16 and the
    low-bit summaries stand for the same vector: scores, masses and lists
    under every rule must agree with the (separately pinned) bf16 path."""
    rng = np.random.default_rng(3)
    P, Hkv, G = 96, 2, 4
    _, means, kb = _pool_of_levels(rng, P, Hkv, bits, step)
    summ = oracle.summaries(kb.reshape(-1, S, D)).reshape(P, Hkv, D)
    assert np.array_equal(bits_to_f64(summ), means)
    codes, steps = oracle.summaries_lowbit(kb.reshape(-1, S, D), bits)
    codes, steps = codes.reshape(P, Hkv, D), steps.reshape(P, Hkv)
    q = bf16_bits(rng.standard_normal((G, D)) * 4.0)
    row = rng.permutation(P).astype(np.int32)
    for L in (P * S, P * S - 5, 40 * S + 3):
        for j in range(Hkv):
            F = L // S
            s_b, m_b = oracle.page_mass(q, summ[row[:F], j], SM)
            s_q, m_q = oracle.page_mass_lowbit(q, codes[row[:F], j], steps[row[:F], j], SM)
            assert np.array_equal(s_b, s_q) and np.array_equal(m_b, m_q)
            for rule, param in ((oracle.RULE_COVERAGE, 0.9), (oracle.RULE_COVERAGE, 0.99),
                                (oracle.RULE_COVERAGE, 1.0), (oracle.RULE_TOPK, 7),
                                (oracle.RULE_TOPDELTA, 0.05)):
                ref = oracle.select_unit_rule(q, summ, j, row, L, rule, param, SM)
                got, _ = oracle.select_unit_lowbit(q, codes, steps, j, row, L, rule, param, SM)
                assert np.array_equal(got, ref), (L, j, rule, param)


def test_scores_within_the_quantisation_bound_and_masses_normalised():
    rng = np.random.default_rng(5)
    F, G = 200, 4
    q_hat = rng.standard_normal(D)
    k = rng.standard_normal((F, S, D))
    k[rng.choice(F, 6, replace=False)] += 2.0 * q_hat
    kb = bf16_bits(k)
    mean = bits_to_f64(kb).mean(axis=1)
    q = bf16_bits(rng.standard_normal((G, D)))
    qf = bits_to_f64(q)
    for bits in (8, 2):
        codes, steps = oracle.summaries_lowbit(kb, bits)
        s, m = oracle.page_mass_lowbit(q, codes, steps, SM)
        exact = SM * qf @ mean.T                                        # [G][F]
        bound = SM * np.abs(qf).sum(axis=1)[:, None] * 0.5 * steps.astype(np.float64)[None, :]
        assert np.all(np.abs(s - exact) <= bound * (1 + 1e-9) + 1e-12)
        assert abs(m.sum() - 1.0) < 1e-12 and np.all(m >= 0)


def test_select_lowbit_tail_permutation_and_dense():
    rng = np.random.default_rng(9)
    P, Hkv, G, bits = 64, 1, 4, 8
    k = rng.standard_normal((P, Hkv, S, D))
    k[5] += 4.0 * rng.standard_normal(D)
    kb = bf16_bits(k)
    codes, steps = oracle.summaries_lowbit(kb.reshape(-1, S, D), bits)
    codes, steps = codes.reshape(P, Hkv, D), steps.reshape(P, Hkv)
    q = bf16_bits(rng.standard_normal((G, D)))
    row = np.arange(P, dtype=np.int32)
    L = 40 * S + 9                                                     # 40 full pages + tail
    lst, mass = oracle.select_unit_lowbit(q, codes, steps, 0, row, L, oracle.RULE_COVERAGE, 0.9, SM)
    assert lst[-1] == 40 and np.all(np.diff(lst) > 0)
    dense, _ = oracle.select_unit_lowbit(q, codes, steps, 0, row, L, oracle.RULE_COVERAGE, 1.0, SM)
    assert np.array_equal(dense, np.arange(41))
    tail_only, _ = oracle.select_unit_lowbit(q, codes, steps, 0, row, 9, oracle.RULE_TOPK, 3, SM)
    assert np.array_equal(tail_only, [0])
    # moving the pages to other physical slots changes nothing
    perm = rng.permutation(P).astype(np.int32)
    codes_p = np.empty_like(codes)
    steps_p = np.empty_like(steps)
    codes_p[perm] = codes
    steps_p[perm] = steps
    lst_p, mass_p = oracle.select_unit_lowbit(q, codes_p, steps_p, 0, perm, L, oracle.RULE_COVERAGE,
                                              0.9, SM)
    assert np.array_equal(lst_p, lst) and np.array_equal(mass_p, mass)
