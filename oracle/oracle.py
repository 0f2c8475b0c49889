"""ctypes binding to the fp64 CPU oracle in ``moira_oracle.c``.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this module.  It shares
no code with the CUDA library and never imports it.

bf16 tensors cross this boundary as numpy ``uint16`` arrays holding the bf16
bit patterns; every computation inside is fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moira_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lib = None

_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i8p = ctypes.POINTER(ctypes.c_int8)
_f32p = ctypes.POINTER(ctypes.c_float)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math) if it is stale."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fno-fast-math", "-shared", "-fPIC",
                        "-std=c11", "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    lib.oracle_round_bf16.argtypes = [ctypes.c_double]
    lib.oracle_round_bf16.restype = ctypes.c_uint16
    lib.oracle_summaries.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, _u16p]
    lib.oracle_summaries.restype = None
    lib.oracle_page_mass.argtypes = [_u16p, _u16p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                     ctypes.c_double, _f64p, _f64p]
    lib.oracle_page_mass.restype = None
    lib.oracle_cover.argtypes = [_f64p, ctypes.c_int32, ctypes.c_double, _u8p, _i32p, _f64p]
    lib.oracle_cover.restype = ctypes.c_int32
    lib.oracle_select_unit.argtypes = [_u16p, _u16p, ctypes.c_int32, ctypes.c_int32, _i32p,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_double, ctypes.c_double, _i32p, _f64p, _i32p, _f64p]
    lib.oracle_select_unit.restype = ctypes.c_int32
    lib.oracle_topk.argtypes = [_f64p, ctypes.c_int32, ctypes.c_int32, _u8p]
    lib.oracle_topk.restype = ctypes.c_int32
    lib.oracle_topdelta.argtypes = [_f64p, ctypes.c_int32, ctypes.c_double, _u8p]
    lib.oracle_topdelta.restype = ctypes.c_int32
    lib.oracle_select_unit_rule.argtypes = [_u16p, _u16p, ctypes.c_int32, ctypes.c_int32, _i32p,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                            ctypes.c_double, _i32p]
    lib.oracle_select_unit_rule.restype = ctypes.c_int32
    lib.oracle_attend_unit.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int32, ctypes.c_int32, _i32p,
                                       _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_double, _f64p]
    lib.oracle_attend_unit.restype = None
    lib.oracle_decode_step.argtypes = [_u16p, _u16p, _u16p, _u16p, _i32p, _i32p,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                       ctypes.c_double, ctypes.c_double, _i32p, _f64p, ctypes.c_int32]
    lib.oracle_decode_step.restype = ctypes.c_int32
    lib.oracle_summaries_lowbit.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, _i8p, _f32p]
    lib.oracle_summaries_lowbit.restype = None
    lib.oracle_page_mass_lowbit.argtypes = [_u16p, _i8p, _f32p, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_double, _f64p, _f64p]
    lib.oracle_page_mass_lowbit.restype = None
    lib.oracle_select_unit_lowbit.argtypes = [_u16p, _i8p, _f32p, ctypes.c_int32, ctypes.c_int32,
                                              _i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32, ctypes.c_double,
                                              ctypes.c_double, _i32p, _f64p]
    lib.oracle_select_unit_lowbit.restype = ctypes.c_int32
    _lib = lib
    return lib


def _c(a: np.ndarray, dtype, ptr):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ptr)


def round_bf16(x: float) -> int:
    """bf16 bit pattern nearest to ``x`` (ties to even)."""
    return int(_load().oracle_round_bf16(float(x)))


def summaries(k_blocks: np.ndarray) -> np.ndarray:
    """Mean key of each block. ``k_blocks``: uint16 [n][S][d] -> uint16 [n][d]."""
    lib = _load()
    n, S, d = k_blocks.shape
    kb, kp = _c(k_blocks, np.uint16, _u16p)
    out = np.empty((n, d), np.uint16)
    lib.oracle_summaries(kp, n, S, d, out.ctypes.data_as(_u16p))
    return out


def page_mass(q_group: np.ndarray, summ: np.ndarray, sm_scale: float):
    """Scores [G][F] and masses [F] of one unit (summaries in logical order)."""
    lib = _load()
    G, d = q_group.shape
    F = summ.shape[0]
    qa, qp = _c(q_group, np.uint16, _u16p)
    sa, sp = _c(summ.reshape(F, d), np.uint16, _u16p)
    scores = np.empty((G, F), np.float64)
    mass = np.empty(F, np.float64)
    lib.oracle_page_mass(qp, sp, G, F, d, float(sm_scale), scores.ctypes.data_as(_f64p),
                         mass.ctypes.data_as(_f64p))
    return scores, mass


def cover(mass: np.ndarray, gamma: float):
    """Coverage rule on given masses: (keep bool [F], k, order [F], cum [F])."""
    lib = _load()
    ma, mp = _c(mass, np.float64, _f64p)
    F = ma.shape[0]
    keep = np.empty(F, np.uint8)
    order = np.empty(F, np.int32)
    cum = np.empty(F, np.float64)
    k = lib.oracle_cover(mp, F, float(gamma), keep.ctypes.data_as(_u8p),
                         order.ctypes.data_as(_i32p), cum.ctypes.data_as(_f64p))
    return keep.astype(bool), int(k), order, cum


def select_unit(q_group, summ_pool, j, page_row, seq_len, gamma, sm_scale, page_size=16):
    """Selection for one unit.

    ``summ_pool``: uint16 [*][Hkv][d] by physical page; ``page_row``: int32
    logical -> physical.  Returns (list of kept LOGICAL pages, mass [F],
    order [F], cum [F]); mass/order/cum are empty when every page is kept
    without estimation (gamma >= 1 or no full page).
    """
    lib = _load()
    G, d = q_group.shape
    Hkv = summ_pool.shape[-2]
    F = seq_len // page_size
    qa, qp = _c(q_group, np.uint16, _u16p)
    sa, sp = _c(summ_pool, np.uint16, _u16p)
    ra, rp = _c(page_row, np.int32, _i32p)
    lst = np.empty(F + 1, np.int32)
    mass = np.zeros(F, np.float64)
    order = np.zeros(F, np.int32)
    cum = np.zeros(F, np.float64)
    n = lib.oracle_select_unit(qp, sp, Hkv, j, rp, seq_len, page_size, G, d, float(gamma),
                               float(sm_scale), lst.ctypes.data_as(_i32p), mass.ctypes.data_as(_f64p),
                               order.ctypes.data_as(_i32p), cum.ctypes.data_as(_f64p))
    return lst[:n].copy(), mass, order, cum


RULE_COVERAGE, RULE_TOPK, RULE_TOPDELTA = 0, 1, 2


def topk(mass: np.ndarray, k: int) -> np.ndarray:
    """Fixed budget: keep mask of the k largest masses (ties: lower index)."""
    lib = _load()
    m = np.ascontiguousarray(mass, np.float64)
    keep = np.zeros(m.shape[0], np.uint8)
    lib.oracle_topk(m.ctypes.data_as(_f64p), m.shape[0], int(k), keep.ctypes.data_as(_u8p))
    return keep.astype(bool)


def topdelta(mass: np.ndarray, delta: float) -> np.ndarray:
    """Relative threshold: keep mask of masses >= delta * max mass."""
    lib = _load()
    m = np.ascontiguousarray(mass, np.float64)
    keep = np.zeros(m.shape[0], np.uint8)
    lib.oracle_topdelta(m.ctypes.data_as(_f64p), m.shape[0], float(delta), keep.ctypes.data_as(_u8p))
    return keep.astype(bool)


def select_unit_rule(q_group, summ_pool, j, page_row, seq_len, rule, param, sm_scale, page_size=16):
    """Selection for one unit under `rule` (RULE_COVERAGE / RULE_TOPK /
    RULE_TOPDELTA with param gamma / k / delta) -> kept LOGICAL pages."""
    lib = _load()
    G, d = q_group.shape
    Hkv = summ_pool.shape[-2]
    F = seq_len // page_size
    qa, qp = _c(q_group, np.uint16, _u16p)
    sa, sp = _c(summ_pool, np.uint16, _u16p)
    ra, rp = _c(page_row, np.int32, _i32p)
    lst = np.empty(F + 1, np.int32)
    n = lib.oracle_select_unit_rule(qp, sp, Hkv, j, rp, seq_len, page_size, G, d, int(rule),
                                    float(param), float(sm_scale), lst.ctypes.data_as(_i32p))
    return lst[:n].copy()


def attend_unit(q_group, k_pool, v_pool, j, page_row, lst, seq_len, sm_scale):
    """Exact fp64 attention of one unit over the listed LOGICAL pages -> [G][d]."""
    lib = _load()
    G, d = q_group.shape
    Hkv, S = k_pool.shape[-3], k_pool.shape[-2]
    qa, qp = _c(q_group, np.uint16, _u16p)
    ka, kp = _c(k_pool, np.uint16, _u16p)
    va, vp = _c(v_pool, np.uint16, _u16p)
    ra, rp = _c(page_row, np.int32, _i32p)
    la, lp = _c(lst, np.int32, _i32p)
    out = np.empty((G, d), np.float64)
    lib.oracle_attend_unit(qp, kp, vp, Hkv, j, rp, lp, la.shape[0], seq_len, S, G, d,
                           float(sm_scale), out.ctypes.data_as(_f64p))
    return out


def decode_step(q, summ, k_pool, v_pool, page_table, seq_lens, gamma, sm_scale, n_threads=0):
    """Select + attend for every (layer, request, KV head) of the given layers.

    q: uint16 [Lyr][B][Hq][d]; summ: uint16 [Lyr][P][Hkv][d];
    k_pool/v_pool: uint16 [Lyr][P][Hkv][S][d]; page_table: int32 [B][max_pages];
    seq_lens: int32 [B].  Returns (lengths [Lyr][B][Hkv], out f64 [Lyr][B][Hq][d],
    threads used).
    """
    lib = _load()
    Lyr, B, Hq, d = q.shape
    P, Hkv, S = k_pool.shape[1], k_pool.shape[2], k_pool.shape[3]
    max_pages = page_table.shape[1]
    qa, qp = _c(q, np.uint16, _u16p)
    sa, sp = _c(summ, np.uint16, _u16p)
    ka, kp = _c(k_pool, np.uint16, _u16p)
    va, vp = _c(v_pool, np.uint16, _u16p)
    ta, tp = _c(page_table, np.int32, _i32p)
    la, lp = _c(seq_lens, np.int32, _i32p)
    lengths = np.empty((Lyr, B, Hkv), np.int32)
    out = np.empty((Lyr, B, Hq, d), np.float64)
    used = lib.oracle_decode_step(qp, sp, kp, vp, tp, lp, Lyr, B, Hq, Hkv, d, S, P, max_pages,
                                  float(gamma), float(sm_scale), lengths.ctypes.data_as(_i32p),
                                  out.ctypes.data_as(_f64p), int(n_threads))
    return lengths, out, int(used)


def summaries_lowbit(k_blocks: np.ndarray, bits: int = 8):
    """Mid-rise low-bit mean key of each block.  ``k_blocks``: uint16
    [n][S][d] -> (codes int8 [n][d], steps float32 [n]); the summary stands
    for (codes + 1/2) * steps."""
    lib = _load()
    n, S, d = k_blocks.shape
    kb, kp = _c(k_blocks, np.uint16, _u16p)
    codes = np.empty((n, d), np.int8)
    steps = np.empty(n, np.float32)
    lib.oracle_summaries_lowbit(kp, n, S, d, int(bits), codes.ctypes.data_as(_i8p),
                                steps.ctypes.data_as(_f32p))
    return codes, steps


def page_mass_lowbit(q_group: np.ndarray, codes: np.ndarray, steps: np.ndarray, sm_scale: float):
    """Scores [G][F] and masses [F] of one unit from low-bit summaries in
    logical order (codes int8 [F][d], steps float32 [F])."""
    lib = _load()
    G, d = q_group.shape
    F = codes.shape[0]
    qa, qp = _c(q_group, np.uint16, _u16p)
    ca, cp = _c(codes.reshape(F, d), np.int8, _i8p)
    sa, sp = _c(steps.reshape(F), np.float32, _f32p)
    scores = np.empty((G, F), np.float64)
    mass = np.empty(F, np.float64)
    lib.oracle_page_mass_lowbit(qp, cp, sp, G, F, d, float(sm_scale), scores.ctypes.data_as(_f64p),
                                mass.ctypes.data_as(_f64p))
    return scores, mass


def select_unit_lowbit(q_group, codes_pool, steps_pool, j, page_row, seq_len, rule, param,
                       sm_scale, page_size=16):
    """Selection for one unit from low-bit summaries under `rule` ->
    (kept LOGICAL pages, mass [F]; zeros when no estimate is made).
    ``codes_pool``: int8 [*][Hkv][d], ``steps_pool``: float32 [*][Hkv], both by
    physical page."""
    lib = _load()
    G, d = q_group.shape
    Hkv = codes_pool.shape[-2]
    F = seq_len // page_size
    qa, qp = _c(q_group, np.uint16, _u16p)
    ca, cp = _c(codes_pool, np.int8, _i8p)
    sa, sp = _c(steps_pool, np.float32, _f32p)
    ra, rp = _c(page_row, np.int32, _i32p)
    lst = np.empty(F + 1, np.int32)
    mass = np.zeros(F, np.float64)
    n = lib.oracle_select_unit_lowbit(qp, cp, sp, Hkv, j, rp, seq_len, page_size, G, d, int(rule),
                                      float(param), float(sm_scale), lst.ctypes.data_as(_i32p),
                                      mass.ctypes.data_as(_f64p))
    return lst[:n].copy(), mass
