"""The comparison rules the GPU parity tests apply to page lists
(helpers.check_list), checked on the CPU against the oracle itself.

The rules accept a list that differs from the oracle's only where fp32 and
fp64 may legitimately decide differently (pages whose cumulative mass meets
the 1e-4 band around gamma, or whose mass ties the cut mass to 1e-6).  A rule
that accepted too much would let a wrong kernel pass, so each plausible kernel
mistake is planted into the oracle's own list (mapped to physical ids, as a
kernel returns it) and must be rejected; the oracle's list itself must pass.
"""
import numpy as np

import helpers as H
from sparse_long_context_page_gb300 import workloads as W


def _unit(seed=0, gamma=0.9):
    sp = W.spec("tiny", layers=1)
    w = W.make_workload(sp, seed=seed, device="cpu")
    ud = H.UnitData(w, 0, 0, 0, with_v=False)
    lst, mass, order, cum = ud.select(gamma)
    phys = ud.phys[np.asarray(lst, np.int64)]
    return ud, np.asarray(lst, np.int64), phys, mass, order, cum


def test_the_oracle_list_passes():
    for gamma in (0.5, 0.9, 0.99):
        ud, lst, phys, *_ = _unit(gamma=gamma)
        assert H.check_list(ud, phys, float(np.float32(gamma))) is None


def test_planted_mistakes_are_rejected():
    gamma = float(np.float32(0.9))
    ud, lst, phys, mass, order, cum = _unit(gamma=gamma)
    F = ud.F
    kept = set(int(x) for x in lst if x < F)
    heaviest = int(order[0])
    assert heaviest in kept
    # a dropped heavy page (an off-by-one in the cut, a lost candidate)
    drop = np.array([p for p in phys if ud.to_logical([p])[0] != heaviest])
    assert H.check_list(ud, drop, gamma) is not None
    # a light page added far below the cut
    light = int(order[-1])
    add = np.sort(np.append(lst, light))
    assert H.check_list(ud, ud.phys[add], gamma) is not None
    # descending order, and a missing tail page
    assert H.check_list(ud, phys[::-1].copy(), gamma) is not None
    if ud.L % 16:
        assert H.check_list(ud, phys[:-1], gamma) is not None
    # a physical id from outside the unit's pages
    bad = phys.copy()
    bad[0] = 10 ** 6
    assert H.check_list(ud, bad, gamma) is not None
    # the right number of pages but the wrong ones: the k lightest instead of the k heaviest
    k = len(kept)
    wrong = np.sort(np.array([int(p) for p in order[-k:]] + ([F] if ud.L % 16 else []), np.int64))
    assert H.check_list(ud, ud.phys[wrong], gamma) is not None


def test_tie_only_excuses_are_counted():
    """A page excused only by the equal-mass clause (not by the gamma band)
    is counted in stats["tie_only"], so the parity tests can bound it."""
    gamma = float(np.float32(0.5))
    ud, lst, phys, mass, order, cum = _unit(gamma=gamma)
    F = ud.F
    k = sum(1 for x in lst if x < F)
    cut = int(order[k - 1])
    # the first page outside the list whose mass equals the cut mass to 1e-6
    # (none in random data): make one by editing the oracle masses seen by
    # check_list, through a unit whose select() returns doctored masses
    twin = int(order[k + 5])
    doctored = mass.copy()
    doctored[twin] = doctored[cut] * (1 + 1e-7)

    class Doctored(H.UnitData):
        def __init__(self, base):
            self.__dict__.update(base.__dict__)

        def select(self, g):
            o = np.argsort(-doctored, kind="stable")
            return lst, doctored, o, np.cumsum(doctored[o])

    du = Doctored(ud)
    swapped = [int(x) for x in lst if x != cut] + [twin]
    swapped = np.sort(np.array(swapped, np.int64))
    stats = {}
    why = H.check_list(du, ud.phys[swapped], gamma, stats)
    assert why is None, why
    assert stats.get("tie_only", 0) >= 1
