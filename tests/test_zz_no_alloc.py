"""moira_select_noalloc: the selection for callers that cannot allocate.

Callers such as plug-ins handed only their input and output buffers, or a
decode loop that must never call cudaMalloc, use this entry point: its
scratch lives in a fixed array inside the library.  It must give exactly the
lists and lengths of moira_select (which uses a caller workspace), call
after call, since both run the same kernels on the same inputs.

This file is named to be collected last; it passes alone in a fresh process
and after the rest of the suite.
"""
import ctypes

import numpy as np
import pytest
import torch

from sparse_long_context_page_gb300 import _binding as mb
from sparse_long_context_page_gb300 import workloads as W
from sparse_long_context_page_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

SCRATCH_BYTES = 4 << 20


def _noalloc(lib, st, l, gamma, lists, lengths):
    w = st.w
    return lib.moira_select_noalloc(
        ctypes.byref(st.shape), w.q[l].data_ptr(), st.summ[l].data_ptr(), st.page_table.data_ptr(),
        st.seq_lens.data_ptr(), w.spec.batch, st.max_pages, float(gamma), float(st.sm_scale),
        lists.data_ptr(), lengths.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,over,gammas", [
    ("tiny", {}, (0.9, 0.99, 1.0)),
    ("llama8b_128k", dict(layers=1), (0.98, 0.99)),
    ("stress_regimes", dict(batch=3, context=(16 * 3000 + 5,)), (0.99,)),
])
def test_noalloc_select_matches_workspace_select(name, over, gammas):
    lib = mb.load_library()
    w = W.make_workload(name, seed=31, device="cuda", **over)
    st = DecodeState(w)
    st.summarize()
    B, Hkv = w.spec.batch, w.spec.kv_heads
    for gamma in gammas:
        g = float(np.float32(gamma))
        ref_lists = torch.full_like(st.lists, -7)
        ref_len = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
        st.select_layer(0, g, ref_lists, ref_len)
        for call in range(2):                       # two calls in a row share the scratch
            lists = torch.full_like(st.lists, -7)
            lengths = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
            assert _noalloc(lib, st, 0, g, lists, lengths) == 0
            torch.cuda.synchronize()
            assert torch.equal(lengths, ref_len), f"{name} gamma {g} call {call}: lengths differ"
            lh, rh, n = lists.cpu().numpy(), ref_lists.cpu().numpy(), ref_len.cpu().numpy()
            for r in range(B):
                for j in range(Hkv):
                    assert np.array_equal(lh[r, j, :n[r, j]], rh[r, j, :n[r, j]]), \
                        f"{name} gamma {g} call {call}: list ({r},{j}) differs"


def test_noalloc_sequence_of_shapes():
    """Calls of different shapes in a row share the one scratch array: a
    large call, then a tiny one whose full-page count is not a multiple of 4
    and whose tail is partial, then the large one again; each gives
    moira_select's lists and lengths."""
    lib = mb.load_library()
    g = float(np.float32(0.99))
    big = W.make_workload("llama8b_128k", seed=41, device="cuda", layers=1, batch=2)
    small = W.make_workload(W.spec("llama8b_128k", batch=3, layers=1, context=(16 * 7 + 5, 16 * 13 + 1, 9)),
                            seed=42, device="cuda")
    states = []
    for w in (big, small):
        st = DecodeState(w)
        st.summarize()
        states.append(st)
    for st in (states[0], states[1], states[0], states[1]):
        B, Hkv = st.batch, st.w.spec.kv_heads
        ref_lists = torch.full_like(st.lists, -7)
        ref_len = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
        st.select_layer(0, g, ref_lists, ref_len)
        lists = torch.full_like(st.lists, -7)
        lengths = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, st, 0, g, lists, lengths) == 0
        torch.cuda.synchronize()
        assert torch.equal(lengths, ref_len)
        lh, rh, n = lists.cpu().numpy(), ref_lists.cpu().numpy(), ref_len.cpu().numpy()
        for r in range(B):
            for j in range(Hkv):
                assert np.array_equal(lh[r, j, :n[r, j]], rh[r, j, :n[r, j]]), (B, r, j)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = mb.load_library()
    w = W.make_workload("tiny", seed=1, device="cuda")
    st = DecodeState(w)
    # 32 requests x 8 query heads x MAX_PAGES_PER_SEQ pages x 4 B of page weights > 4 MiB
    nb = 32
    big = nb * 8 * mb.MAX_PAGES_PER_SEQ * 4
    assert big > SCRATCH_BYTES
    pt = torch.zeros((nb, mb.MAX_PAGES_PER_SEQ), dtype=torch.int32, device="cuda")
    sl = torch.zeros(nb, dtype=torch.int32, device="cuda")
    lists = torch.zeros((nb, 2, mb.MAX_PAGES_PER_SEQ), dtype=torch.int32, device="cuda")
    lengths = torch.zeros((nb, 2), dtype=torch.int32, device="cuda")
    rc = lib.moira_select_noalloc(ctypes.byref(st.shape), w.q[0].data_ptr(), st.summ[0].data_ptr(),
                                  pt.data_ptr(), sl.data_ptr(), nb, mb.MAX_PAGES_PER_SEQ, 0.9,
                                  float(st.sm_scale), lists.data_ptr(), lengths.data_ptr(), None)
    assert rc == 4                                  # MOIRA_EUNSUPPORTED, nothing launched
