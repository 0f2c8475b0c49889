"""Shared test plumbing: host copies of one unit's data for the oracle, and
the comparison rules for page lists and attention outputs.

Comparison rules (all derived from the selection's definition, stated here
once):
  * lists are compared as sets of LOGICAL pages; a page in the symmetric
    difference of the CUDA and oracle sets is accepted only when it sits at
    the gamma boundary: its oracle cumulative-mass interval [C_before,
    C_through] meets [gamma - 1e-4, gamma + 1e-4], or its oracle mass equals
    the oracle's cut mass to 1e-6 relative (fp32 vs fp64 reordering of
    near-equal masses; the tests count the pages only this second clause
    excuses and bound them, TIE_ONLY_MAX per test);
  * the CUDA set must still cover gamma under the oracle's masses (to 1e-4);
  * lengths must match exactly unless the oracle's running sum crosses gamma
    within 1e-4 of it; then they may differ by at most the number of pages
    whose cumulative-mass interval meets the band (one, unless the masses at
    the cut are below 1e-4, as in the flat tail of gamma near 1);
  * structure: ascending logical order, the partial tail page last;
  * attention output (fp32) within max-abs 1e-2 and relative L2 1e-3 per
    (request, query head) row (bf16 inputs, fp32 accumulation).
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle

BAND = 1e-4
TIE_REL = 1e-6
TIE_ONLY_MAX = 8          # pages per test that only the equal-mass clause may excuse
MAX_ABS = 1e-2
REL_L2 = 1e-3


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class UnitData:
    """Host copy of one (layer, request, KV head) unit in logical page order."""

    def __init__(self, w, l: int, r: int, j: int, with_v: bool = True, fmt: int = 0):
        S = w.spec.page_size
        self.fmt = fmt                     # summary format: 0 bf16, 1 eight-bit, 2 two-bit
        G = w.group
        self.L = int(w.seq_lens[r])
        self.n = self.L // S + (self.L % S != 0)
        self.F = self.L // S
        row = torch.from_numpy(w.page_table[r, :self.n].astype(np.int64)).to(w.k_pool.device)
        self.phys = w.page_table[r, :self.n].astype(np.int64)
        self.q = u16(w.q[l, r, j * G:(j + 1) * G])                         # [G][d]
        self.k = u16(w.k_pool[l].index_select(0, row)[:, j])              # [n][S][d]
        self.v = u16(w.v_pool[l].index_select(0, row)[:, j]) if with_v else None
        self.sm_scale = w.sm_scale
        self._summ = None
        self._lowbit = None

    @property
    def summ(self):
        if self._summ is None:
            self._summ = oracle.summaries(self.k[:self.F]) if self.F else np.zeros((0, 128), np.uint16)
        return self._summ

    @property
    def lowbit(self):
        """Oracle low-bit summaries of the full pages: (codes [F][d], steps [F])."""
        if self._lowbit is None:
            bits = 8 if self.fmt == 1 else 2
            if self.F:
                self._lowbit = oracle.summaries_lowbit(self.k[:self.F], bits)
            else:
                self._lowbit = (np.zeros((0, 128), np.int8), np.zeros(0, np.float32))
        return self._lowbit

    def select(self, gamma: float):
        """Oracle selection: (logical list, mass, order, cum), from the
        summaries of this unit's format."""
        rows = np.arange(max(self.F, 1), dtype=np.int32)
        if self.fmt == 0:
            pool = self.summ[:, None, :] if self.F else np.zeros((1, 1, 128), np.uint16)
            return oracle.select_unit(self.q, pool, 0, rows, self.L, gamma, self.sm_scale)
        codes, steps = self.lowbit
        if not self.F:
            codes, steps = np.zeros((1, 128), np.int8), np.zeros(1, np.float32)
        lst, mass = oracle.select_unit_lowbit(self.q, codes[:, None, :], steps[:, None], 0, rows,
                                              self.L, oracle.RULE_COVERAGE, gamma, self.sm_scale)
        if gamma >= 1.0 or self.F == 0:
            z = np.zeros(self.F)
            return lst, z, np.zeros(self.F, np.int32), z
        _, _, order, cum = oracle.cover(mass, gamma)
        return lst, mass, order, cum

    def attend(self, logical_list) -> np.ndarray:
        return oracle.attend_unit(self.q, self.k[:, None], self.v[:, None], 0,
                                  np.arange(max(self.n, 1), dtype=np.int32),
                                  np.asarray(logical_list, np.int32), self.L, self.sm_scale)

    def to_logical(self, phys_list) -> np.ndarray:
        inv = {int(p): i for i, p in enumerate(self.phys)}
        return np.array([inv.get(int(p), -1) for p in phys_list], np.int64)


def check_list(ud: UnitData, gpu_phys: np.ndarray, gamma: float, stats: dict | None = None) -> str | None:
    """None if the CUDA list is acceptable against the oracle, else a reason.
    With `stats`, stats["tie_only"] counts the differing pages that only the
    equal-mass clause (not the gamma band) excuses."""
    lg = ud.to_logical(gpu_phys)
    if np.any(lg < 0):
        return f"unknown physical page ids {gpu_phys[lg < 0][:5]}"
    if len(lg) > 1 and np.any(np.diff(lg) <= 0):
        return "list not in ascending logical order"
    tail = ud.L % 16 != 0
    if tail and (len(lg) == 0 or lg[-1] != ud.F):
        return "partial tail page missing or not last"
    o_list, mass, order, cum = ud.select(gamma)
    if gamma >= 1.0 or ud.F == 0:
        return None if np.array_equal(lg, o_list) else f"dense list differs ({len(lg)} vs {len(o_list)})"
    full_g = set(int(x) for x in lg if x < ud.F)
    full_o = set(int(x) for x in o_list if x < ud.F)
    k = len(full_o)
    rank = np.empty(ud.F, np.int64)
    rank[order] = np.arange(ud.F)
    m_cut = mass[order[k - 1]]
    bad = []
    for p in full_g ^ full_o:
        j = rank[p]
        c_before = cum[j - 1] if j > 0 else 0.0
        c_thru = cum[j]
        near_band = c_before <= gamma + BAND and c_thru >= gamma - BAND
        near_tie = abs(mass[p] - m_cut) <= TIE_REL * max(m_cut, 1e-30)
        if not (near_band or near_tie):
            bad.append((p, j, c_before, c_thru, mass[p]))
        elif near_tie and not near_band and stats is not None:
            stats["tie_only"] = stats.get("tie_only", 0) + 1
    if bad:
        return f"{len(bad)} pages differ away from the boundary, e.g. {bad[:3]} (k={k})"
    covered = mass[list(full_g)].sum() if full_g else 0.0
    if covered < gamma - BAND and not (cum[-1] < gamma):
        return f"CUDA set covers only {covered:.6f} < gamma {gamma}"
    if len(full_g) != k:
        c_km1 = cum[k - 2] if k >= 2 else 0.0
        near = abs(cum[k - 1] - gamma) <= BAND or abs(c_km1 - gamma) <= BAND
        before = np.concatenate([[0.0], cum[:-1]])
        in_band = int(np.count_nonzero((before <= gamma + BAND) & (cum >= gamma - BAND)))
        if not near or abs(len(full_g) - k) > max(1, in_band):
            return f"length {len(full_g)} vs oracle {k} (C_k-1={c_km1:.7f}, C_k={cum[k-1]:.7f})"
    return None


def out_errors(got: np.ndarray, ref: np.ndarray):
    """(max-abs, worst per-row relative L2) over rows of the last axis."""
    got = np.asarray(got, np.float64).reshape(-1, ref.shape[-1])
    ref = np.asarray(ref, np.float64).reshape(-1, ref.shape[-1])
    max_abs = float(np.max(np.abs(got - ref))) if got.size else 0.0
    num = np.linalg.norm(got - ref, axis=1)
    den = np.linalg.norm(ref, axis=1)
    rel = np.where(den > 0, num / np.maximum(den, 1e-300), num)
    return max_abs, float(rel.max()) if rel.size else 0.0


# Width of the fp32-vs-fp64 band for the alternative rules: a page may be
# decided differently only when its oracle mass is within RULE_BAND
# (relative) of the rule's boundary mass (the k-th largest mass, or delta *
# the largest mass), or when both are below RULE_FLOOR: fp32 masses of that
# size underflow in the chunk-relative products, so their order is not kept
# (a fixed budget larger than the pages that carry any mass ends among them).
RULE_BAND = 1e-5
RULE_FLOOR = 1e-30


def check_rule_list(ud: UnitData, gpu_phys: np.ndarray, rule: int, param: float) -> str | None:
    """None if the CUDA list under top-k / top-delta is acceptable against the
    oracle rule applied to the oracle masses, else a reason."""
    lg = ud.to_logical(gpu_phys)
    if np.any(lg < 0):
        return f"unknown physical page ids {gpu_phys[lg < 0][:5]}"
    if len(lg) > 1 and np.any(np.diff(lg) <= 0):
        return "list not in ascending logical order"
    tail = ud.L % 16 != 0
    if tail and (len(lg) == 0 or lg[-1] != ud.F):
        return "partial tail page missing or not last"
    if ud.F == 0:
        return None if len(lg) == int(tail) else "pages listed for an empty context"
    _, mass, order, _ = ud.select(0.5)
    full_g = set(int(x) for x in lg if x < ud.F)
    if rule == oracle.RULE_TOPK:
        keep = oracle.topk(mass, int(param))
        k = min(int(param), ud.F)
        if len(full_g) != k:
            return f"top-k kept {len(full_g)} full pages, want {k}"
        edge = mass[order[k - 1]] if k > 0 else 0.0
    else:
        keep = oracle.topdelta(mass, param)
        edge = param * mass.max()
    full_o = set(int(x) for x in np.flatnonzero(keep))
    bad = [p for p in full_g ^ full_o
           if abs(mass[p] - edge) > RULE_BAND * edge and max(mass[p], edge) > RULE_FLOOR]
    if bad:
        return f"{len(bad)} pages decided differently away from the boundary, e.g. {bad[:3]}"
    return None


def pack_lowbit(codes: np.ndarray, steps: np.ndarray, bits: int, rec_bytes: int) -> np.ndarray:
    """Oracle codes [P][Hkv][d] and steps [P][Hkv] laid out as the library's
    per-page records (include/moira.h): KV heads in groups of min(Hkv, 4);
    per group the heads' codes (one int8 each for 8 bits; element i at bits
    2*(i%4) of byte i/4, as code + 2, for 2 bits), then their fp32 steps,
    then zero padding to 16 bytes past the codes."""
    P, Hkv, d = codes.shape
    gh = min(Hkv, 4)
    cb = d * bits // 8
    if bits == 8:
        packed = codes.view(np.uint8)                                   # [P][Hkv][cb]
    else:
        u = (codes.astype(np.int16) + 2).astype(np.uint8).reshape(P, Hkv, cb, 4)
        packed = u[..., 0] | (u[..., 1] << 2) | (u[..., 2] << 4) | (u[..., 3] << 6)
    gbytes = gh * cb + 16
    out = np.zeros((P, rec_bytes), np.uint8)
    st = np.ascontiguousarray(steps, np.float32).view(np.uint8).reshape(P, Hkv, 4)
    for g in range(Hkv // gh):
        o = g * gbytes
        out[:, o:o + gh * cb] = packed[:, g * gh:(g + 1) * gh].reshape(P, gh * cb)
        out[:, o + gh * cb:o + gh * cb + 4 * gh] = st[:, g * gh:(g + 1) * gh].reshape(P, 4 * gh)
    return out
