"""The C ABI without a GPU: the library builds and loads, exports every
function include/moira.h declares, and its host-side checks reject bad
arguments before any CUDA call (fake, never-dereferenced pointers)."""
import ctypes
import os
import re

import pytest

import sparse_long_context_page_gb300 as moira
from sparse_long_context_page_gb300 import _binding as mb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000          # 64 KiB-aligned fake device address; never dereferenced


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moira.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moira_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    lib = moira.load_library()
    decl = declared_functions()
    assert len(decl) >= 10
    for name in decl:
        assert hasattr(lib, name), f"{name} declared in moira.h but not exported"
    assert set(decl) == set(mb.EXPORTS)


def test_load_balance_build_exports_the_timing_entry():
    """The load-balance build exports everything libmoira.so does plus
    moira_set_cta_times (include/moira_cta_times.h); libmoira.so has none of it.
    Its host checks reject a missing buffer before any CUDA call."""
    from sparse_long_context_page_gb300 import build
    text = open(os.path.join(ROOT, "include", "moira_cta_times.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    extra = set(re.findall(r"\b(moira_[a-z_]+)\s*\(", text))
    assert extra == {"moira_set_cta_times"}
    moira.load_library()
    timed = ctypes.CDLL(build.LIB_CTA_TIMES)
    for name in list(mb.EXPORTS) + sorted(extra):
        assert hasattr(timed, name), name
    assert not hasattr(moira.load_library(), "moira_set_cta_times")
    timed.moira_set_cta_times.argtypes = [ctypes.c_void_p, ctypes.c_int32]
    assert timed.moira_set_cta_times(None, 3) == 1
    assert timed.moira_set_cta_times(FAKE, -1) == 1
    assert timed.moira_set_cta_times(None, 0) == 0


def test_status_strings():
    lib = moira.load_library()
    for code in range(5):
        assert lib.moira_status_string(code)
    assert lib.moira_status_string(99) == b"unknown status"


def _select(lib, shape, gamma=0.9, sm=0.088, q=FAKE, batch=1, max_pages=64):
    return lib.moira_select(ctypes.byref(shape), q, FAKE, FAKE, FAKE, batch, max_pages, gamma, sm,
                            FAKE, FAKE, FAKE, 1 << 30, None)


def test_select_rejects_bad_arguments_on_host():
    lib = moira.load_library()
    ok = moira.Shape.of(32, 8, 1024)
    assert _select(lib, ok, gamma=0.0) == 1
    assert _select(lib, ok, gamma=1.5) == 1
    assert _select(lib, ok, gamma=float("nan")) == 1
    assert _select(lib, ok, sm=-1.0) == 1
    assert _select(lib, ok, sm=float("inf")) == 1
    assert _select(lib, ok, q=0) == 1                         # null pointer
    assert _select(lib, ok, q=FAKE + 2) == 1                  # misaligned
    assert _select(lib, ok, batch=0) == 1
    assert _select(lib, ok, max_pages=mb.MAX_PAGES_PER_SEQ + 1) == 4
    assert _select(lib, ok, batch=mb.MAX_UNITS // 8 + 1) == 4
    assert _select(lib, moira.Shape.of(32, 8, 1024, head_dim=64)) == 4
    assert _select(lib, moira.Shape.of(32, 8, 1024, page_size=32)) == 4
    assert _select(lib, moira.Shape.of(16, 8, 1024)) == 4     # group of 2
    assert _select(lib, moira.Shape.of(30, 8, 1024)) == 1     # not a multiple
    assert _select(lib, moira.Shape.of(32, 8, 0)) == 1
    assert _select(lib, moira.Shape.of(32, 8, 1 << 25)) == 4  # TMA rows beyond 2^31


def test_select_rule_rejects_bad_rules_and_params_on_host():
    lib = moira.load_library()
    ok = moira.Shape.of(32, 8, 1024)

    def call(rule, param, sm=0.088):
        return lib.moira_select_rule(ctypes.byref(ok), FAKE, FAKE, FAKE, FAKE, 2, 64, rule, param, sm,
                                     FAKE, FAKE, FAKE, 1 << 30, None)

    for rule, param in [(3, 0.5), (-1, 0.5),                               # unknown rule
                        (mb.RULE_COVERAGE, 0.0), (mb.RULE_COVERAGE, 1.5),
                        (mb.RULE_COVERAGE, float("nan")),
                        (mb.RULE_TOPK, -1.0), (mb.RULE_TOPK, 2.5),           # not a whole count
                        (mb.RULE_TOPK, float(1 << 25)), (mb.RULE_TOPK, float("inf")),
                        (mb.RULE_TOPDELTA, 0.0), (mb.RULE_TOPDELTA, 1.01),
                        (mb.RULE_TOPDELTA, float("nan"))]:
        assert call(rule, param) == 1, (rule, param)
    assert call(mb.RULE_TOPK, 3.0, sm=0.0) == 1


def test_append_kv_rejects_bad_arguments_on_host():
    lib = moira.load_library()
    ok = moira.Shape.of(32, 8, 1024)

    def call(shape=ok, k=FAKE, v=FAKE, kp=FAKE, vp=FAKE, summ=FAKE, pt=FAKE, sl=FAKE, batch=2, max_pages=64):
        return lib.moira_append_kv(ctypes.byref(shape), k, v, kp, vp, summ, pt, sl, batch, max_pages, None)

    assert call(k=0) == 1 and call(summ=0) == 1 and call(sl=0) == 1     # null pointers
    assert call(kp=FAKE + 4) == 1                                       # misaligned
    assert call(batch=0) == 1
    assert call(max_pages=mb.MAX_PAGES_PER_SEQ + 1) == 4
    assert call(shape=moira.Shape.of(32, 8, 1024, head_dim=64)) == 4


def test_diag_wait_timeout_rejects_bad_arguments_on_host():
    lib = moira.load_library()
    assert lib.moira_diag_wait_timeout(None, 1 << 20, 1000, None) == 1
    assert lib.moira_diag_wait_timeout(FAKE, 16, 1000, None) == 1        # smaller than the status block
    assert lib.moira_diag_wait_timeout(FAKE, 1 << 20, 0, None) == 1
    assert lib.moira_diag_wait_timeout(FAKE, 1 << 20, 10 ** 10 + 1, None) == 1


def test_attend_and_step_reject_bad_arguments_on_host():
    lib = moira.load_library()
    ok = moira.Shape.of(32, 8, 1024)
    sp = ctypes.byref(ok)
    assert lib.moira_attend(sp, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 0.0, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.moira_attend(sp, FAKE, FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 64, 0.1, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.moira_attend(sp, FAKE, FAKE, 0, FAKE, FAKE, FAKE, 1, 64, 0.1, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.moira_decode_step(sp, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 0.9, 0.1,
                                 FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.moira_decode_step(sp, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64, 1.01, 0.1,
                                 FAKE, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.moira_update_summaries(sp, FAKE, FAKE, FAKE, -1, None) == 1
    assert lib.moira_update_summaries(sp, FAKE, FAKE + 4, FAKE, 3, None) == 1
    assert lib.moira_update_summaries(sp, FAKE, FAKE, FAKE, 0, None) == 0      # nothing to do
    assert lib.moira_workspace_init(None, 100, None) == 2
    st = ctypes.c_uint32(0)
    assert lib.moira_read_device_status(None, 1024, ctypes.byref(st), 0, None) == 2
    assert lib.moira_workspace_bytes(ctypes.byref(moira.Shape.of(30, 8, 16)), 1, 64) == 0


def test_binding_rejects_host_tensors():
    torch = pytest.importorskip("torch")
    shape = moira.Shape.of(8, 2, 16)
    t = torch.zeros(4, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        moira.update_summaries(shape, t, t, torch.zeros(1, dtype=torch.int32))


@pytest.mark.parametrize("hkv,bf16,q8,q2", [(1, 256, 144, 48), (2, 512, 272, 80), (4, 1024, 528, 144),
                                            (8, 2048, 1056, 288)])
def test_summary_page_bytes_follow_the_record_layout(hkv, bf16, q8, q2):
    """Hkv * d * 2 bytes for bf16; Hkv * d * b / 8 code bytes plus Hkv fp32
    steps, padded to 16 bytes, for the low-bit formats."""
    lib = moira.load_library()
    shape = moira.Shape.of(4 * hkv, hkv, 1024)
    got = [lib.moira_summary_page_bytes(ctypes.byref(shape), f)
           for f in (mb.SUMM_BF16, mb.SUMM_Q8, mb.SUMM_Q2)]
    assert got == [bf16, q8, q2]
    assert lib.moira_summary_page_bytes(ctypes.byref(shape), 3) == 0
    assert lib.moira_summary_page_bytes(ctypes.byref(moira.Shape.of(30, 8, 16)), mb.SUMM_Q8) == 0


def test_format_entry_points_reject_bad_arguments_on_host():
    lib = moira.load_library()
    ok = moira.Shape.of(32, 8, 1024)
    sp = ctypes.byref(ok)
    for fmt in (-1, 3):
        assert lib.moira_update_summaries_ex(sp, fmt, FAKE, FAKE, FAKE, 4, None) == 1
        assert lib.moira_append_kv_ex(sp, fmt, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 2, 64, None) == 1
        assert lib.moira_select_ex(sp, fmt, FAKE, FAKE, FAKE, FAKE, 1, 64, mb.RULE_COVERAGE, 0.9, 0.1,
                                   FAKE, FAKE, FAKE, 1 << 30, None) == 1
        assert lib.moira_decode_step_ex(sp, fmt, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64,
                                        mb.RULE_COVERAGE, 0.9, 0.1, FAKE, FAKE, FAKE, FAKE, 1 << 30,
                                        None) == 1
    q8 = mb.SUMM_Q8
    assert lib.moira_update_summaries_ex(sp, q8, FAKE, FAKE + 8, FAKE, 4, None) == 1     # misaligned
    assert lib.moira_update_summaries_ex(sp, q8, FAKE, FAKE, FAKE, 0, None) == 0         # nothing to do
    assert lib.moira_select_ex(sp, q8, FAKE, FAKE, FAKE, FAKE, 1, 64, mb.RULE_TOPK, 2.5, 0.1,
                               FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert lib.moira_select_ex(sp, q8, FAKE, FAKE, FAKE, FAKE, 1, mb.MAX_PAGES_PER_SEQ + 1,
                               mb.RULE_COVERAGE, 0.9, 0.1, FAKE, FAKE, FAKE, 1 << 30, None) == 4
    assert lib.moira_decode_step_ex(sp, q8, 2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 64,
                                    mb.RULE_TOPDELTA, 0.0, 0.1, FAKE, FAKE, FAKE, FAKE, 1 << 30,
                                    None) == 1


def test_select_noalloc_rejects_what_select_rejects_on_host():
    """moira_select_noalloc shares moira_select's argument checks: the same
    bad arguments give the same codes, before any CUDA call."""
    lib = moira.load_library()
    ok = moira.Shape.of(32, 8, 1024)

    def noalloc(shape=ok, q=FAKE, summ=FAKE, gamma=0.9, sm=0.088, batch=1, max_pages=64, lists=FAKE):
        return lib.moira_select_noalloc(ctypes.byref(shape), q, summ, FAKE, FAKE, batch, max_pages, gamma,
                                        sm, lists, FAKE, None)

    cases = [dict(gamma=0.0), dict(gamma=1.5), dict(gamma=float("nan")), dict(sm=-1.0),
             dict(sm=float("inf")), dict(q=0), dict(lists=0), dict(q=FAKE + 2), dict(summ=FAKE + 8),
             dict(batch=0), dict(max_pages=mb.MAX_PAGES_PER_SEQ + 1), dict(batch=mb.MAX_UNITS // 8 + 1),
             dict(shape=moira.Shape.of(32, 8, 1024, head_dim=64)), dict(shape=moira.Shape.of(16, 8, 1024)),
             dict(shape=moira.Shape.of(30, 8, 1024)), dict(shape=moira.Shape.of(32, 8, 0)),
             dict(shape=moira.Shape.of(32, 8, 1 << 25))]
    for kw in cases:
        sel = _select(lib, kw.get("shape", ok), gamma=kw.get("gamma", 0.9), sm=kw.get("sm", 0.088),
                      q=kw.get("q", FAKE), batch=kw.get("batch", 1), max_pages=kw.get("max_pages", 64))
        got = noalloc(**kw)
        assert got in (1, 4), (kw, got)
        if not ({"lists", "summ"} & kw.keys()):
            assert got == sel, (kw, got, sel)


def test_select_clustered_rejects_what_select_rejects_on_host():
    """moira_select_clustered shares moira_select's argument checks, and
    moira_select_cluster_size answers 0 for invalid arguments."""
    lib = moira.load_library()
    ok = moira.Shape.of(32, 8, 1024)

    def clustered(shape=ok, q=FAKE, gamma=0.9, sm=0.088, batch=1, max_pages=64):
        return lib.moira_select_clustered(ctypes.byref(shape), q, FAKE, FAKE, FAKE, batch, max_pages, gamma, sm,
                                          FAKE, FAKE, FAKE, 1 << 30, None)

    for kw in [dict(gamma=0.0), dict(gamma=1.5), dict(gamma=float("nan")), dict(sm=-1.0), dict(q=0),
               dict(q=FAKE + 2), dict(batch=0), dict(max_pages=mb.MAX_PAGES_PER_SEQ + 1),
               dict(shape=moira.Shape.of(32, 8, 1024, head_dim=64)), dict(shape=moira.Shape.of(30, 8, 1024))]:
        sel = _select(lib, kw.get("shape", ok), gamma=kw.get("gamma", 0.9), sm=kw.get("sm", 0.088),
                      q=kw.get("q", FAKE), batch=kw.get("batch", 1), max_pages=kw.get("max_pages", 64))
        assert clustered(**kw) == sel, kw
    assert lib.moira_select_cluster_size(ctypes.byref(moira.Shape.of(30, 8, 1024)), 1, 64) == 0
    assert lib.moira_select_cluster_size(ctypes.byref(ok), 0, 64) == 0
