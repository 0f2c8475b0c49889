"""The coverage selection in one launch (moira_select_clustered: one
thread-block cluster per list).

It must give moira_select's lists and lengths (page scores into the
workspace, then the cut, in two launches) bit for bit, since both use the
same estimator arithmetic, the same fixed-order normaliser and the same exact
integer cut, and every list must pass the oracle's comparison rules.  Sizes span one and two rounds of chunks per
block, ragged tails, the empty and single-page
cases, crossing bins of every size (pairwise, one warp, and the 256-bin
passes over all blocks' masses when more pages tie than the candidate list
holds).
"""
import numpy as np
import pytest
import torch

import helpers as H
from sparse_long_context_page_gb300 import _binding as mb
from sparse_long_context_page_gb300 import workloads as W
from sparse_long_context_page_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _state(w, max_pages=None):
    st = DecodeState(w, max_pages=max_pages)
    st.summarize()
    return st


def _compare(w, st, l, gamma, check_oracle=True, stats=None):
    """moira_select_clustered against moira_select, bit for bit, and
    (optionally) every unit against the oracle."""
    B, Hkv = w.spec.batch, w.spec.kv_heads
    assert mb.select_cluster_size(st.shape, B, st.max_pages) in (8, 16)
    lists = torch.full_like(st.lists, -7)
    lengths = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    st.select_layer_clustered(l, gamma, lists, lengths)
    ref_lists = torch.full_like(st.lists, -7)
    ref_len = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    st.select_layer(l, gamma, ref_lists, ref_len)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    assert torch.equal(lengths, ref_len), f"layer {l} gamma {gamma}: lengths differ from moira_select's"
    lh, rh, nh = lists.cpu().numpy(), ref_lists.cpu().numpy(), ref_len.cpu().numpy()
    for r in range(B):
        for j in range(Hkv):
            n = nh[r, j]
            assert np.array_equal(lh[r, j, :n], rh[r, j, :n]), f"layer {l} gamma {gamma}: list ({r},{j}) differs"
            assert np.all(lh[r, j, n:] == -7), f"({r},{j}): written past its length"
    if check_oracle:
        for r in range(B):
            for j in range(Hkv):
                ud = H.UnitData(w, l, r, j, with_v=False)
                why = H.check_list(ud, lh[r, j, :nh[r, j]], gamma, stats)
                assert why is None, f"layer {l} req {r} kv {j} gamma {gamma}: {why}"
    return lh, nh


@pytest.mark.parametrize("name,over,gammas", [
    ("tiny", {}, (0.5, 0.9, 0.99)),
    ("llama8b_32k", dict(layers=2), (0.99,)),
    ("llama8b_128k", dict(layers=2), (0.98, 0.99, 0.999)),
    ("serving_ragged", dict(batch=1, layers=2), (0.99,)),
    ("stress_regimes", dict(batch=1, context=(16 * 4000 + 7,)), (0.99, 0.9)),
])
def test_clustered_select_matches_select_and_oracle(name, over, gammas):
    w = W.make_workload(name, seed=21, device="cuda", **over)
    st = _state(w)
    stats = {}
    for l in range(w.spec.layers):
        for g in gammas:
            _compare(w, st, l, float(np.float32(g)), stats=stats)
    assert stats.get("tie_only", 0) <= H.TIE_ONLY_MAX, stats


def test_clustered_select_limits():
    """Which batches the one-launch form takes: a request of up to 8192 pages
    (16 chunks per block at cluster size 8 need two rounds of 16).  More lists
    than the device holds clusters at once, or more pages, return
    MOIRA_EUNSUPPORTED and launch nothing."""
    sh = mb.Shape.of(32, 8, 1 << 20)
    assert mb.select_cluster_size(sh, 1, 8192) in (8, 16)
    assert mb.select_cluster_size(sh, 1, 16384) == 0
    assert mb.select_cluster_size(sh, 64, 8192) == 0
    sp = W.spec("llama8b_128k", batch=1, layers=1, context=(16 * 16383 + 11,))
    w = W.make_workload(sp, seed=17, device="cuda")
    st = _state(w)
    lists = torch.full_like(st.lists, -7)
    with pytest.raises(mb.MoiraError) as e:
        st.select_layer_clustered(0, float(np.float32(0.99)), lists, torch.zeros_like(st.lengths[0]))
    assert e.value.status == 4
    torch.cuda.synchronize()
    assert bool((lists == -7).all())


def test_clustered_select_two_rounds_at_the_limit():
    """8192 pages, the largest request that takes one launch: every block
    scores two rounds of 16 chunks at cluster size 8."""
    sp = W.spec("llama8b_128k", batch=1, layers=1, context=(16 * 8191 + 11,))
    w = W.make_workload(sp, seed=17, device="cuda")
    st = _state(w)
    for g in (0.9, 0.99):
        _compare(w, st, 0, float(np.float32(g)))


def test_clustered_select_edge_lengths():
    """Empty, sub-page, exact-page, one-chunk, ragged and multi-chunk
    contexts, max_pages beyond the request's need; gamma down to 1e-6 (one
    page) and up to just below 1."""
    for L in (0, 1, 15, 16, 17, 16 * 31 + 3, 16 * 32, 16 * 33 + 1, 16 * 257 + 3, 16 * 5000):
        sp = W.spec("llama8b_128k", batch=1, layers=1, context=(L,))
        w = W.make_workload(sp, seed=5, device="cuda")
        st = _state(w, max_pages=w.max_pages + 37)
        for g in (1e-6, 0.5, 0.99, 0.99999):
            _compare(w, st, 0, float(np.float32(g)))


@pytest.mark.parametrize("F", [50, 500, 3000, 8000])
def test_clustered_select_all_masses_tied(F):
    """Identical keys: every mass is equal.  50 and 500 pages take the
    pairwise and one-warp refinements; 3000 and 8000 exceed the candidate list
    and take the 256-bin passes over every block's masses.  The ceil(gamma*F)
    lowest pages are kept, as moira_select keeps."""
    L = 16 * F + 5
    sp = W.spec("llama8b_128k", batch=1, layers=1, context=(L,))
    w = W.make_workload(sp, seed=9, device="cuda")
    key = torch.randn(128, generator=torch.Generator(device="cuda").manual_seed(1), device="cuda")
    w.k_pool[:] = key.to(torch.bfloat16)
    st = _state(w)
    for gamma in (0.3, 0.7, 0.9, 0.99):
        g = float(np.float32(gamma))
        lh, nh = _compare(w, st, 0, g, check_oracle=False)
        if abs(g * F - round(g * F)) > 1e-3:
            k = int(np.ceil(g * F))
            for j in range(w.spec.kv_heads):
                ud = H.UnitData(w, 0, 0, j, with_v=False)
                logical = ud.to_logical(lh[0, j, :nh[0, j]])
                assert list(logical) == list(range(k)) + [F], f"F={F} gamma={g}: {len(logical)} vs {k}+1"


def test_clustered_select_graph_replays_equal_moira_select():
    """The layers' clustered selections captured in one graph and replayed
    give moira_select's lists and lengths bit for bit on every replay."""
    w = W.make_workload("llama8b_128k", seed=2, device="cuda", layers=3)
    st = _state(w)
    g32 = float(np.float32(0.99))
    L = w.spec.layers
    lists = torch.zeros((L,) + tuple(st.lists.shape), dtype=torch.int32, device="cuda")
    lengths = torch.zeros_like(st.lengths)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for l in range(L):
            st.select_layer_clustered(l, g32, lists[l], lengths[l])
        with torch.cuda.graph(graph, stream=s):
            for l in range(L):
                st.select_layer_clustered(l, g32, lists[l], lengths[l])
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        lists.zero_()
        lengths.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert st.device_status() == 0
        for l in range(L):
            ref_lists = torch.zeros_like(st.lists)
            ref_len = torch.zeros_like(st.lengths[l])
            st.select_layer(l, g32, ref_lists, ref_len)
            torch.cuda.synchronize()
            assert torch.equal(lengths[l], ref_len), f"layer {l}: lengths differ"
            n = ref_len.cpu().numpy()
            a, b = lists[l].cpu().numpy(), ref_lists.cpu().numpy()
            for j in range(w.spec.kv_heads):
                assert np.array_equal(a[0, j, :n[0, j]], b[0, j, :n[0, j]]), f"layer {l} list {j}"


def test_bad_page_ids_are_reported_and_skipped():
    """A page id outside the pool is not read: the status word reports it,
    and the other lists still equal moira_select's."""
    sp = W.spec("llama8b_128k", batch=1, layers=1, context=(16 * 700 + 3,))
    w = W.make_workload(sp, seed=8, device="cuda")
    st = _state(w)
    st.page_table[0, 123] = w.num_phys_pages + 5
    g = float(np.float32(0.9))
    lists = torch.zeros_like(st.lists)
    lengths = torch.zeros((1, w.spec.kv_heads), dtype=torch.int32, device="cuda")
    st.select_layer_clustered(0, g, lists, lengths)
    torch.cuda.synchronize()
    assert st.device_status() & mb.DEV_BADPAGE
    mb.workspace_init(st.ws)
    ref_lists = torch.zeros_like(st.lists)
    ref_len = torch.zeros_like(lengths)
    st.select_layer(0, g, ref_lists, ref_len)
    torch.cuda.synchronize()
    assert st.device_status() & mb.DEV_BADPAGE
    assert torch.equal(lengths, ref_len)
    for j in range(w.spec.kv_heads):
        n = int(ref_len[0, j])
        assert torch.equal(lists[0, j, :n], ref_lists[0, j, :n])
