"""ctypes binding over ``libmoira.so`` (argument marshalling only).

Every function takes torch CUDA tensors, checks dtype / device / layout,
and passes raw pointers plus the current CUDA stream to the C ABI declared in
``include/moira.h``.  All computation happens in the library's kernels; there
is no CPU or PyTorch fallback: if the library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

from . import build as _build

_lib = None

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_u32p = ctypes.POINTER(ctypes.c_uint32)

STATUS = {0: "MOIRA_OK", 1: "MOIRA_EINVAL", 2: "MOIRA_EWORKSPACE", 3: "MOIRA_ECUDA",
          4: "MOIRA_EUNSUPPORTED"}
DEV_BADPAGE, DEV_BADLEN, DEV_TIMEOUT = 0x1, 0x2, 0x4
HEAD_DIM, PAGE_SIZE, GROUP = 128, 16, 4
MAX_PAGES_PER_SEQ, MAX_UNITS = 16384, 4096

# every symbol include/moira.h declares
EXPORTS = ("moira_workspace_bytes", "moira_workspace_init", "moira_update_summaries",
           "moira_select", "moira_attend", "moira_decode_step", "moira_decode_step_host",
           "moira_read_device_status", "moira_attend_grid_blocks", "moira_status_string",
           "moira_select_noalloc", "moira_select_rule", "moira_append_kv",
           "moira_diag_wait_timeout", "moira_summary_page_bytes", "moira_update_summaries_ex",
           "moira_append_kv_ex", "moira_select_ex", "moira_decode_step_ex", "moira_select_attend",
           "moira_select_attend_ex", "moira_select_attend_is_fused", "moira_score_ex", "moira_diag_wait_chain",
           "moira_diag_barrier_timeout", "moira_select_clustered", "moira_select_cluster_size")

# page rules of moira_select_rule (moira_rule in include/moira.h)
RULE_COVERAGE, RULE_TOPK, RULE_TOPDELTA = 0, 1, 2
# page-summary formats (moira_summ_format in include/moira.h)
SUMM_BF16, SUMM_Q8, SUMM_Q2 = 0, 1, 2


class MoiraError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} "
                         f"({_lib.moira_status_string(status).decode() if _lib else ''})")


class Shape(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_phys_pages", ctypes.c_int64)]

    @classmethod
    def of(cls, num_q_heads, num_kv_heads, num_phys_pages, head_dim=HEAD_DIM, page_size=PAGE_SIZE):
        return cls(num_q_heads, num_kv_heads, head_dim, page_size, num_phys_pages)


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Load libmoira.so (building it in-tree first when it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(f"{path} is missing; build it with sparse_long_context_page_gb300.build")
        _build.build()
    _lib = _declare(ctypes.CDLL(path))
    return _lib


@contextlib.contextmanager
def library_variant(path: str):
    """Route every call of this module through another build of the library
    (e.g. the load-balance build, build.LIB_CTA_TIMES) inside the block."""
    global _lib
    saved = load_library()
    _lib = _declare(ctypes.CDLL(path))
    try:
        yield _lib
    finally:
        _lib = saved


def _declare(lib):
    """Argument and result types of the C ABI on a loaded library."""
    sp = ctypes.POINTER(Shape)
    lib.moira_workspace_bytes.argtypes = [sp, _i32, _i32]
    lib.moira_workspace_bytes.restype = ctypes.c_size_t
    lib.moira_workspace_init.argtypes = [_vp, ctypes.c_size_t, _vp]
    lib.moira_workspace_init.restype = ctypes.c_int
    lib.moira_update_summaries.argtypes = [sp, _vp, _vp, _vp, _i32, _vp]
    lib.moira_append_kv.argtypes = [sp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp]
    lib.moira_append_kv.restype = ctypes.c_int
    lib.moira_update_summaries.restype = ctypes.c_int
    lib.moira_select.argtypes = [sp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float, ctypes.c_float,
                                 _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.moira_select.restype = ctypes.c_int
    lib.moira_select_rule.argtypes = [sp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, ctypes.c_float,
                                      ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.moira_select_rule.restype = ctypes.c_int
    lib.moira_attend.argtypes = [sp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float, _vp,
                                 _vp, ctypes.c_size_t, _vp]
    lib.moira_attend.restype = ctypes.c_int
    lib.moira_decode_step.argtypes = [sp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                      ctypes.c_float, ctypes.c_float, _vp, _vp, _vp, _vp,
                                      ctypes.c_size_t, _vp]
    lib.moira_decode_step.restype = ctypes.c_int
    lib.moira_decode_step_host.argtypes = [sp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                           ctypes.c_float, ctypes.c_float, _vp, _vp, _vp, _vp, _vp,
                                           ctypes.c_size_t, _vp]
    lib.moira_decode_step_host.restype = ctypes.c_int
    lib.moira_read_device_status.argtypes = [_vp, ctypes.c_size_t, _u32p, _i32, _vp]
    lib.moira_diag_wait_timeout.argtypes = [_vp, ctypes.c_size_t, ctypes.c_uint64, _vp]
    lib.moira_diag_wait_timeout.restype = ctypes.c_int
    lib.moira_read_device_status.restype = ctypes.c_int
    lib.moira_attend_grid_blocks.argtypes = []
    lib.moira_attend_grid_blocks.restype = _i32
    lib.moira_select_noalloc.argtypes = [sp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float,
                                         ctypes.c_float, _vp, _vp, _vp]
    lib.moira_select_noalloc.restype = ctypes.c_int
    lib.moira_summary_page_bytes.argtypes = [sp, _i32]
    lib.moira_summary_page_bytes.restype = ctypes.c_size_t
    lib.moira_update_summaries_ex.argtypes = [sp, _i32, _vp, _vp, _vp, _i32, _vp]
    lib.moira_update_summaries_ex.restype = ctypes.c_int
    lib.moira_append_kv_ex.argtypes = [sp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _vp]
    lib.moira_append_kv_ex.restype = ctypes.c_int
    lib.moira_select_ex.argtypes = [sp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, _i32, ctypes.c_float,
                                    ctypes.c_float, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.moira_select_ex.restype = ctypes.c_int
    lib.moira_decode_step_ex.argtypes = [sp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                         _i32, ctypes.c_float, ctypes.c_float, _vp, _vp, _vp, _vp,
                                         ctypes.c_size_t, _vp]
    lib.moira_decode_step_ex.restype = ctypes.c_int
    lib.moira_select_attend.argtypes = [sp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float,
                                        ctypes.c_float, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.moira_select_attend.restype = ctypes.c_int
    lib.moira_select_attend_ex.argtypes = [sp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32,
                                           ctypes.c_float, ctypes.c_float, _vp, _vp, _vp, _vp,
                                           ctypes.c_size_t, _vp]
    lib.moira_select_attend_ex.restype = ctypes.c_int
    lib.moira_score_ex.argtypes = [sp, _i32, _vp, _vp, _vp, _vp, _i32, _i32, ctypes.c_float, _vp,
                                   ctypes.c_size_t, _vp]
    lib.moira_score_ex.restype = ctypes.c_int
    lib.moira_select_attend_is_fused.argtypes = [sp, _i32, _i32]
    lib.moira_select_attend_is_fused.restype = _i32
    lib.moira_select_clustered.argtypes = lib.moira_select.argtypes
    lib.moira_select_clustered.restype = ctypes.c_int
    lib.moira_select_cluster_size.argtypes = [sp, _i32, _i32]
    lib.moira_select_cluster_size.restype = _i32
    lib.moira_diag_wait_chain.argtypes = [_vp, ctypes.c_size_t, ctypes.c_uint64, _i32, _vp]
    lib.moira_diag_wait_chain.restype = ctypes.c_int
    lib.moira_diag_barrier_timeout.argtypes = [_vp, ctypes.c_size_t, ctypes.c_uint64, _i32, _vp]
    lib.moira_diag_barrier_timeout.restype = ctypes.c_int
    lib.moira_status_string.argtypes = [ctypes.c_int]
    lib.moira_status_string.restype = ctypes.c_char_p
    if hasattr(lib, "moira_set_cta_times"):          # the load-balance build
        lib.moira_set_cta_times.argtypes = [_vp, _i32]
        lib.moira_set_cta_times.restype = ctypes.c_int
    return lib


def _check(st: int, what: str):
    if st != 0:
        raise MoiraError(st, what)


def _stream(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dev(t: torch.Tensor, name: str, dtype, ndim=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    return t.data_ptr()


def shape_of(num_q_heads: int, num_kv_heads: int, num_phys_pages: int) -> Shape:
    return Shape.of(num_q_heads, num_kv_heads, num_phys_pages)


def workspace_bytes(shape: Shape, batch: int, max_pages: int) -> int:
    n = load_library().moira_workspace_bytes(ctypes.byref(shape), batch, max_pages)
    if n == 0:
        raise MoiraError(1, "moira_workspace_bytes")
    return int(n)


def make_workspace(shape: Shape, batch: int, max_pages: int, device=None) -> torch.Tensor:
    """Allocate (through torch) and zero a workspace for these sizes."""
    n = workspace_bytes(shape, batch, max_pages)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    workspace_init(ws)
    return ws


def workspace_init(ws: torch.Tensor, stream=None):
    _check(load_library().moira_workspace_init(_dev(ws, "workspace", torch.uint8), ws.numel(),
                                               _stream(stream)), "moira_workspace_init")


def summary_page_bytes(shape: Shape, fmt: int = SUMM_BF16) -> int:
    """Bytes of one physical page's summaries (all KV heads) in format `fmt`."""
    n = load_library().moira_summary_page_bytes(ctypes.byref(shape), int(fmt))
    if n == 0:
        raise MoiraError(1, "moira_summary_page_bytes")
    return int(n)


def make_summaries(shape: Shape, fmt: int = SUMM_BF16, layers: int | None = None, device=None):
    """Zeroed summary buffer(s) for `fmt`: bf16 [(layers,) P, Hkv, d] for
    SUMM_BF16, else uint8 [(layers,) P, page_bytes] records."""
    lead = () if layers is None else (layers,)
    P = shape.num_phys_pages
    if fmt == SUMM_BF16:
        return torch.zeros(lead + (P, shape.num_kv_heads, shape.head_dim), dtype=torch.bfloat16,
                           device=device or "cuda")
    return torch.zeros(lead + (P, summary_page_bytes(shape, fmt)), dtype=torch.uint8,
                       device=device or "cuda")


def _summ(summ: torch.Tensor, fmt: int):
    return _dev(summ, "summ", torch.bfloat16 if fmt == SUMM_BF16 else torch.uint8)


def update_summaries(shape: Shape, k_pool: torch.Tensor, summ: torch.Tensor,
                     phys_pages: torch.Tensor, stream=None, fmt: int = SUMM_BF16):
    """Summaries of every listed physical page p from k_pool[p]'s keys: the
    bf16 mean key (SUMM_BF16) or its low-bit record (SUMM_Q8 / SUMM_Q2)."""
    lib = load_library()
    pp = _dev(phys_pages, "phys_pages", torch.int32, 1)
    if fmt == SUMM_BF16:
        st = lib.moira_update_summaries(ctypes.byref(shape), _dev(k_pool, "k_pool", torch.bfloat16),
                                        _summ(summ, fmt), pp, phys_pages.numel(), _stream(stream))
    else:
        st = lib.moira_update_summaries_ex(ctypes.byref(shape), int(fmt),
                                           _dev(k_pool, "k_pool", torch.bfloat16), _summ(summ, fmt),
                                           pp, phys_pages.numel(), _stream(stream))
    _check(st, "moira_update_summaries")


def append_kv(shape: Shape, k_new, v_new, k_pool, v_pool, summ, page_table, seq_lens, stream=None,
              fmt: int = SUMM_BF16):
    """Write each request's new token (token seq_lens[r]-1) into its page and
    recompute the summary (in format `fmt`) of every page that this fills."""
    lib = load_library()
    batch, max_pages = page_table.shape
    args = (_dev(k_new, "k_new", torch.bfloat16), _dev(v_new, "v_new", torch.bfloat16),
            _dev(k_pool, "k_pool", torch.bfloat16), _dev(v_pool, "v_pool", torch.bfloat16),
            _summ(summ, fmt), _dev(page_table, "page_table", torch.int32, 2),
            _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages, _stream(stream))
    if fmt == SUMM_BF16:
        st = lib.moira_append_kv(ctypes.byref(shape), *args)
    else:
        st = lib.moira_append_kv_ex(ctypes.byref(shape), int(fmt), *args)
    _check(st, "moira_append_kv")


def select(shape: Shape, q, summ, page_table, seq_lens, gamma: float, sm_scale: float, lists,
           lengths, ws, stream=None):
    """Per-(request, KV head) coverage lists for one layer (see include/moira.h)."""
    lib = load_library()
    batch, max_pages = page_table.shape
    _check(lib.moira_select(ctypes.byref(shape), _dev(q, "q", torch.bfloat16),
                            _dev(summ, "summ", torch.bfloat16),
                            _dev(page_table, "page_table", torch.int32, 2),
                            _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages,
                            float(gamma), float(sm_scale), _dev(lists, "lists", torch.int32),
                            _dev(lengths, "lengths", torch.int32), _dev(ws, "workspace", torch.uint8),
                            ws.numel(), _stream(stream)), "moira_select")


def select_clustered(shape: Shape, q, summ, page_table, seq_lens, gamma: float, sm_scale: float, lists,
                     lengths, ws, stream=None):
    """moira_select in its one-launch cluster form (moira_select_clustered):
    the same lists and lengths; raises MoiraError(MOIRA_EUNSUPPORTED) when the
    batch does not fit the device's clusters."""
    lib = load_library()
    batch, max_pages = page_table.shape
    _check(lib.moira_select_clustered(ctypes.byref(shape), _dev(q, "q", torch.bfloat16),
                                      _dev(summ, "summ", torch.bfloat16),
                                      _dev(page_table, "page_table", torch.int32, 2),
                                      _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages,
                                      float(gamma), float(sm_scale), _dev(lists, "lists", torch.int32),
                                      _dev(lengths, "lengths", torch.int32), _dev(ws, "workspace", torch.uint8),
                                      ws.numel(), _stream(stream)), "moira_select_clustered")


def select_cluster_size(shape: Shape, batch: int, max_pages: int) -> int:
    """Cluster size (16 or 8) of moira_select_clustered for these sizes, 0 if unsupported."""
    return int(load_library().moira_select_cluster_size(ctypes.byref(shape), int(batch), int(max_pages)))


def select_rule(shape: Shape, q, summ, page_table, seq_lens, rule: int, param: float,
                sm_scale: float, lists, lengths, ws, stream=None):
    """Per-(request, KV head) lists for one layer under a page rule:
    RULE_COVERAGE (param = gamma), RULE_TOPK (param = k) or RULE_TOPDELTA
    (param = delta); see include/moira.h."""
    lib = load_library()
    batch, max_pages = page_table.shape
    _check(lib.moira_select_rule(ctypes.byref(shape), _dev(q, "q", torch.bfloat16),
                                 _dev(summ, "summ", torch.bfloat16),
                                 _dev(page_table, "page_table", torch.int32, 2),
                                 _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages,
                                 int(rule), float(param), float(sm_scale),
                                 _dev(lists, "lists", torch.int32), _dev(lengths, "lengths", torch.int32),
                                 _dev(ws, "workspace", torch.uint8), ws.numel(), _stream(stream)),
           "moira_select_rule")


def select_ex(shape: Shape, fmt: int, q, summ, page_table, seq_lens, rule: int, param: float,
              sm_scale: float, lists, lengths, ws, stream=None):
    """select_rule reading summaries in format `fmt` (SUMM_BF16 / SUMM_Q8 /
    SUMM_Q2); see include/moira.h."""
    lib = load_library()
    batch, max_pages = page_table.shape
    _check(lib.moira_select_ex(ctypes.byref(shape), int(fmt), _dev(q, "q", torch.bfloat16),
                               _summ(summ, fmt), _dev(page_table, "page_table", torch.int32, 2),
                               _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages,
                               int(rule), float(param), float(sm_scale),
                               _dev(lists, "lists", torch.int32), _dev(lengths, "lengths", torch.int32),
                               _dev(ws, "workspace", torch.uint8), ws.numel(), _stream(stream)),
           "moira_select_ex")


def select_attend(shape: Shape, q, summ, k_pool, v_pool, page_table, seq_lens, gamma: float,
                  sm_scale: float, lists, lengths, out, ws, stream=None, fmt: int = SUMM_BF16):
    """One layer's coverage selection and attention (moira_select_attend /
    _ex): the lists and lengths of select(), the output of attend() over them."""
    lib = load_library()
    batch, max_pages = page_table.shape
    args = (_dev(q, "q", torch.bfloat16), _summ(summ, fmt), _dev(k_pool, "k_pool", torch.bfloat16),
            _dev(v_pool, "v_pool", torch.bfloat16), _dev(page_table, "page_table", torch.int32, 2),
            _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages, float(gamma), float(sm_scale),
            _dev(lists, "lists", torch.int32), _dev(lengths, "lengths", torch.int32),
            _dev(out, "out", torch.float32), _dev(ws, "workspace", torch.uint8), ws.numel(), _stream(stream))
    if fmt == SUMM_BF16:
        st = lib.moira_select_attend(ctypes.byref(shape), *args)
    else:
        st = lib.moira_select_attend_ex(ctypes.byref(shape), int(fmt), *args)
    _check(st, "moira_select_attend")


def score(shape: Shape, q, summ, page_table, seq_lens, sm_scale: float, ws, stream=None,
          fmt: int = SUMM_BF16):
    """The page-scoring kernel alone (moira_score_ex): results stay in the
    workspace; for timing how a layer's work splits."""
    lib = load_library()
    batch, max_pages = page_table.shape
    _check(lib.moira_score_ex(ctypes.byref(shape), int(fmt), _dev(q, "q", torch.bfloat16), _summ(summ, fmt),
                              _dev(page_table, "page_table", torch.int32, 2),
                              _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages, float(sm_scale),
                              _dev(ws, "workspace", torch.uint8), ws.numel(), _stream(stream)),
           "moira_score_ex")


def select_attend_is_fused(shape: Shape, batch: int, max_pages: int) -> bool:
    """Whether select_attend takes its single-launch form for these sizes."""
    return bool(load_library().moira_select_attend_is_fused(ctypes.byref(shape), int(batch), int(max_pages)))


def attend(shape: Shape, q, k_pool, v_pool, lists, lengths, seq_lens, max_pages: int,
           sm_scale: float, out, ws, stream=None):
    """Attention of one layer over the listed pages; writes fp32 ``out``."""
    lib = load_library()
    batch = seq_lens.numel()
    _check(lib.moira_attend(ctypes.byref(shape), _dev(q, "q", torch.bfloat16),
                            _dev(k_pool, "k_pool", torch.bfloat16), _dev(v_pool, "v_pool", torch.bfloat16),
                            _dev(lists, "lists", torch.int32), _dev(lengths, "lengths", torch.int32),
                            _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages,
                            float(sm_scale), _dev(out, "out", torch.float32),
                            _dev(ws, "workspace", torch.uint8), ws.numel(), _stream(stream)),
           "moira_attend")


def decode_step(shape: Shape, q_all, k_pool_all, v_pool_all, summ_all, page_table, seq_lens,
                gamma: float, sm_scale: float, lists, lengths_all, out_all, ws, stream=None):
    """select + attend for every layer, in order on one stream."""
    lib = load_library()
    batch, max_pages = page_table.shape
    _check(lib.moira_decode_step(ctypes.byref(shape), q_all.shape[0],
                                 _dev(q_all, "q_all", torch.bfloat16),
                                 _dev(k_pool_all, "k_pool_all", torch.bfloat16),
                                 _dev(v_pool_all, "v_pool_all", torch.bfloat16),
                                 _dev(summ_all, "summ_all", torch.bfloat16),
                                 _dev(page_table, "page_table", torch.int32, 2),
                                 _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages,
                                 float(gamma), float(sm_scale), _dev(lists, "lists", torch.int32),
                                 _dev(lengths_all, "lengths_all", torch.int32),
                                 _dev(out_all, "out_all", torch.float32),
                                 _dev(ws, "workspace", torch.uint8), ws.numel(), _stream(stream)),
           "moira_decode_step")


def decode_step_ex(shape: Shape, fmt: int, q_all, k_pool_all, v_pool_all, summ_all, page_table,
                   seq_lens, rule: int, param: float, sm_scale: float, lists, lengths_all, out_all,
                   ws, stream=None):
    """decode_step with summaries in format `fmt` and any page rule."""
    lib = load_library()
    batch, max_pages = page_table.shape
    _check(lib.moira_decode_step_ex(ctypes.byref(shape), int(fmt), q_all.shape[0],
                                    _dev(q_all, "q_all", torch.bfloat16),
                                    _dev(k_pool_all, "k_pool_all", torch.bfloat16),
                                    _dev(v_pool_all, "v_pool_all", torch.bfloat16),
                                    _summ(summ_all, fmt),
                                    _dev(page_table, "page_table", torch.int32, 2),
                                    _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages,
                                    int(rule), float(param), float(sm_scale),
                                    _dev(lists, "lists", torch.int32),
                                    _dev(lengths_all, "lengths_all", torch.int32),
                                    _dev(out_all, "out_all", torch.float32),
                                    _dev(ws, "workspace", torch.uint8), ws.numel(), _stream(stream)),
           "moira_decode_step_ex")


def decode_step_host(shape: Shape, q_host, q_dev, k_pool_all, v_pool_all, summ_all, page_table,
                     seq_lens, gamma: float, sm_scale: float, lists, lengths_all, out_dev,
                     out_host, ws, stream=None):
    """The step with q read from and out written to HOST (pinned) tensors."""
    lib = load_library()
    for t, nm in ((q_host, "q_host"), (out_host, "out_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous host tensor")
    if q_host.dtype != torch.bfloat16 or out_host.dtype != torch.float32:
        raise TypeError("q_host must be bf16 and out_host fp32")
    batch, max_pages = page_table.shape
    _check(lib.moira_decode_step_host(ctypes.byref(shape), q_host.shape[0], q_host.data_ptr(),
                                      _dev(q_dev, "q_dev", torch.bfloat16),
                                      _dev(k_pool_all, "k_pool_all", torch.bfloat16),
                                      _dev(v_pool_all, "v_pool_all", torch.bfloat16),
                                      _dev(summ_all, "summ_all", torch.bfloat16),
                                      _dev(page_table, "page_table", torch.int32, 2),
                                      _dev(seq_lens, "seq_lens", torch.int32, 1), batch, max_pages,
                                      float(gamma), float(sm_scale),
                                      _dev(lists, "lists", torch.int32),
                                      _dev(lengths_all, "lengths_all", torch.int32),
                                      _dev(out_dev, "out_dev", torch.float32), out_host.data_ptr(),
                                      _dev(ws, "workspace", torch.uint8), ws.numel(),
                                      _stream(stream)), "moira_decode_step_host")


def read_device_status(ws, clear: bool = True, stream=None) -> int:
    """Synchronise the stream and return the MOIRA_DEV_* bits (host call)."""
    lib = load_library()
    out = ctypes.c_uint32(0)
    _check(lib.moira_read_device_status(_dev(ws, "workspace", torch.uint8), ws.numel(),
                                        ctypes.byref(out), 1 if clear else 0, _stream(stream)),
           "moira_read_device_status")
    return int(out.value)


def diag_wait_timeout(ws, limit_ns: int, stream=None):
    """Launch the bounded-wait diagnostic: a wait that runs out after
    ``limit_ns`` and sets DEV_TIMEOUT in the workspace status word."""
    lib = load_library()
    _check(lib.moira_diag_wait_timeout(_dev(ws, "workspace", torch.uint8), ws.numel(), int(limit_ns),
                                       _stream(stream)), "moira_diag_wait_timeout")


def diag_wait_chain(ws, limit_ns: int, n_waits: int, stream=None):
    """Launch the give-up diagnostic: n_waits waits on barriers nothing
    completes; the first runs out after ``limit_ns``, the rest give up at once."""
    lib = load_library()
    _check(lib.moira_diag_wait_chain(_dev(ws, "workspace", torch.uint8), ws.numel(), int(limit_ns),
                                     int(n_waits), _stream(stream)), "moira_diag_wait_chain")


def diag_barrier_timeout(ws, limit_ns: int, blocks: int, stream=None):
    """Launch the inter-block barrier diagnostic: ``blocks`` blocks meet at a
    barrier that never completes and give up after ``limit_ns``."""
    lib = load_library()
    _check(lib.moira_diag_barrier_timeout(_dev(ws, "workspace", torch.uint8), ws.numel(), int(limit_ns),
                                          int(blocks), _stream(stream)), "moira_diag_barrier_timeout")


def set_cta_times(buf, max_launches: int):
    """Load-balance build only (inside library_variant(build.LIB_CTA_TIMES)):
    the next max_launches attention launches record each block's (start, end)
    %globaltimer ns into buf, int64 [max_launches][grid blocks][2] on the
    device; None, 0 stops recording."""
    lib = load_library()
    if not hasattr(lib, "moira_set_cta_times"):
        raise RuntimeError("set_cta_times needs the load-balance build (build.LIB_CTA_TIMES)")
    ptr = None if buf is None else _dev(buf, "cta_times", torch.int64)
    _check(lib.moira_set_cta_times(ptr, int(max_launches)), "moira_set_cta_times")


def attend_grid_blocks() -> int:
    return int(load_library().moira_attend_grid_blocks())
