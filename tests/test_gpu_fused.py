"""The single-launch selection + attention of small batches (moira_select_attend).

Its lists and lengths must equal moira_select's bit for bit (the same
estimator arithmetic and the same exact cut, spread over many blocks), its
output must equal moira_attend's over those lists bit for bit (the same plan
and data path), and it must match the oracle's attention over those lists
for every (request, KV head) unit.  The decode step runs it per layer, so a step must
equal the per-layer calls bit for bit.  Sizes keep the oracle at seconds
while spanning many selecting blocks per list, ragged tails, crowded
crossing bins and the empty and single-page cases.
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


def _state(name, seed=0, max_pages=None, **over):
    w = W.make_workload(name, seed=seed, device="cuda", **over)
    st = DecodeState(w, max_pages=max_pages)
    st.summarize()
    return w, st


def _fused_layer(w, st, l, gamma, check_oracle=True):
    """select_attend on layer l against select (bit for bit) and the oracle
    (every unit).  Returns the number of units checked."""
    assert mb.select_attend_is_fused(st.shape, w.spec.batch, st.max_pages)
    B, Hkv, G = w.spec.batch, w.spec.kv_heads, w.group
    lists = torch.full_like(st.lists, -7)
    lengths = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    out = torch.full_like(st.out[l], 7.0)
    st.select_attend_layer(l, gamma, lists, lengths, out)
    ref_lists = torch.full_like(st.lists, -7)
    ref_len = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
    st.select_layer(l, gamma, ref_lists, ref_len)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    assert torch.equal(lengths, ref_len), f"layer {l} gamma {gamma}: lengths differ from moira_select"
    lh, rh, nh, oh = lists.cpu().numpy(), ref_lists.cpu().numpy(), ref_len.cpu().numpy(), out.cpu().numpy()
    for r in range(B):
        for j in range(Hkv):
            n = nh[r, j]
            assert np.array_equal(lh[r, j, :n], rh[r, j, :n]), f"layer {l} gamma {gamma}: list ({r},{j}) differs"
    # the attention is k_attend's plan and data path over the same lists
    ref_out = torch.full_like(st.out[l], 7.0)
    st.attend_layer(l, ref_lists, ref_len, ref_out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out), f"layer {l} gamma {gamma}: output differs from moira_attend's"
    if not check_oracle:
        return 0
    for r in range(B):
        for j in range(Hkv):
            ud = H.UnitData(w, l, r, j)
            gl = lh[r, j, :nh[r, j]]
            why = H.check_list(ud, gl, gamma)
            assert why is None, f"layer {l} req {r} kv {j} gamma {gamma}: {why}"
            lg = ud.to_logical(gl)
            if len(lg) == 0:
                assert np.all(oh[r, j * G:(j + 1) * G] == 0.0), f"r{r} j{j}: empty list not zero"
                continue
            ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ud.attend(lg))
            assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"l{l} r{r} j{j}: max-abs {ma:.3g} rel-L2 {rl:.3g}"
    return B * Hkv


@pytest.mark.parametrize("name,over,gammas", [
    ("tiny", {}, (0.9, 0.99, 1.0)),
    ("llama8b_32k", dict(layers=1), (0.99,)),
    ("llama8b_128k", dict(layers=1), (0.98, 0.99, 1.0)),
    ("serving_ragged", dict(batch=2, layers=1), (0.99,)),
    ("stress_regimes", dict(batch=2, context=(16 * 4000 + 7,)), (0.99,)),
    ("stress_regimes", dict(batch=7, context=(16 * 1200 + 3,)), (0.99, 0.5)),
])
def test_select_attend_matches_select_and_oracle(name, over, gammas):
    w, st = _state(name, seed=13, **over)
    for g in gammas:
        assert _fused_layer(w, st, 0, float(np.float32(g))) == w.spec.batch * w.spec.kv_heads


def test_select_attend_edge_lengths():
    """Empty, sub-page, exact-page and tail-only contexts in one ragged batch
    (7 requests, 56 lists), with max_pages larger than any request needs."""
    sp = W.spec("llama8b_128k", batch=7, layers=1, context=(0, 1, 15, 16, 17, 16 * 33, 16 * 257 + 3))
    w = W.make_workload(sp, seed=5, device="cuda")
    st = DecodeState(w, max_pages=w.max_pages + 37)
    st.summarize()
    for gamma in (1e-6, 0.5, 0.99, 1.0):
        _fused_layer(w, st, 0, float(np.float32(gamma)))


@pytest.mark.parametrize("F", [50, 500, 3000])
def test_select_attend_all_masses_tied(F):
    """Identical keys: every mass is equal, so the crossing bin holds every
    page; 3000 pages exceed the candidate list and take the global 256-bin
    levels.  The ceil(gamma*F) lowest pages are kept, as moira_select keeps."""
    L = 16 * F + 5
    sp = W.spec("llama8b_128k", batch=1, layers=1, context=(L,))
    w = W.make_workload(sp, seed=9, device="cuda")
    key = torch.randn(128, generator=torch.Generator(device="cuda").manual_seed(1), device="cuda")
    w.k_pool[:] = key.to(torch.bfloat16)
    st = DecodeState(w)
    st.summarize()
    for gamma in (0.3, 0.7, 0.9, 0.99):
        g = float(np.float32(gamma))
        _fused_layer(w, st, 0, g)
        lists, lengths, _ = st.select_attend_layer(0, g)
        torch.cuda.synchronize()
        if abs(g * F - round(g * F)) > 1e-3:
            k = int(np.ceil(g * F))
            for j in range(w.spec.kv_heads):
                ud = H.UnitData(w, 0, 0, j, with_v=False)
                logical = ud.to_logical(lists[0, j, :lengths[0, j]].cpu().numpy())
                assert list(logical) == list(range(k)) + [F], f"F={F} gamma={g}: {len(logical)} vs {k}+1"


def test_select_attend_longest_context():
    """One request of 16383 full pages and a tail (256k tokens), 2 layers."""
    w, st = _state("llama8b_128k", seed=17, layers=2, context=(16 * 16383 + 11,))
    for l in range(2):
        _fused_layer(w, st, l, float(np.float32(0.99)))


def test_decode_step_equals_select_attend_per_layer():
    """The decode step is the per-layer moira_select_attend, bit for bit
    (from layer 1 on the score kernel reads the page table early)."""
    w, st = _state("llama8b_32k", seed=50, layers=4, context=(16 * 900 + 5,))
    gamma = float(np.float32(0.99))
    st.step(gamma)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    out_s, len_s = st.out.clone(), st.lengths.clone()
    for l in range(w.spec.layers):
        lists = torch.full_like(st.lists, -1)
        lengths = torch.zeros_like(st.lengths[l])
        out = torch.zeros_like(st.out[l])
        st.select_attend_layer(l, gamma, lists, lengths, out)
        torch.cuda.synchronize()
        assert torch.equal(lengths, len_s[l]), f"layer {l}: lengths differ"
        assert torch.equal(out, out_s[l]), f"layer {l}: outputs differ"
    assert st.device_status() == 0


def test_fused_graph_replays_are_bit_identical():
    """The 128k step captured once and replayed three times gives the eager
    step's lengths and outputs bit for bit: the cut uses exact integer sums
    and the merges a fixed order, whatever order the blocks arrive in."""
    w, st = _state("llama8b_128k", seed=2, layers=3)
    g32 = float(np.float32(0.99))
    st.step(g32)
    torch.cuda.synchronize()
    out_e, len_e = st.out.clone(), st.lengths.clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st.step(g32)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        st.out.zero_()
        st.lengths.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(st.lengths, len_e)
        assert torch.equal(st.out, out_e)
    assert st.device_status() == 0


def test_larger_batches_take_the_two_launch_form():
    """64 lists or more, or more pages per selecting block than one block
    takes, run moira_select then moira_attend; the call gives the same
    lists as moira_select either way."""
    w, st = _state("serving_ragged", seed=3, batch=8, layers=1)
    assert not mb.select_attend_is_fused(st.shape, 8, st.max_pages)
    g = float(np.float32(0.99))
    lists, lengths, out = st.select_attend_layer(0, g)
    ref_lists = torch.zeros_like(st.lists)
    ref_len = torch.zeros_like(lengths)
    st.select_layer(0, g, ref_lists, ref_len)
    torch.cuda.synchronize()
    assert torch.equal(lengths, ref_len)
    assert st.device_status() == 0


def test_a_barrier_that_never_completes_is_reported():
    """The inter-block barrier of the single-launch form, sized for one block
    more than the grid: every block gives up after the limit (20 ms), the
    status word holds MOIRA_DEV_TIMEOUT, and the workspace, cleared and
    re-initialised, then serves a correct fused layer."""
    import time
    w, st = _state("tiny", seed=0)
    assert st.device_status() == 0
    t0 = time.perf_counter()
    mb.diag_barrier_timeout(st.ws, 20_000_000, 32)
    status = mb.read_device_status(st.ws)
    took = time.perf_counter() - t0
    assert status & mb.DEV_TIMEOUT, hex(status)
    assert 0.015 < took < 2.0, took
    mb.workspace_init(st.ws)
    _fused_layer(w, st, 0, float(np.float32(0.9)))
    assert st.device_status() == 0


def test_waits_give_up_once_per_launch():
    """64 waits in a row on barriers nothing completes, 20 ms limit each: the
    first runs out and the rest give up at once, so the launch ends in well
    under 64 x 20 ms, reports MOIRA_DEV_TIMEOUT, and the context stays usable."""
    import time
    w, st = _state("tiny", seed=0)
    t0 = time.perf_counter()
    mb.diag_wait_chain(st.ws, 20_000_000, 64)
    status = mb.read_device_status(st.ws)
    took = time.perf_counter() - t0
    assert status & mb.DEV_TIMEOUT, hex(status)
    assert took < 0.2, took
    mb.workspace_init(st.ws)
    st.step(float(np.float32(0.99)))
    torch.cuda.synchronize()
    assert st.device_status() == 0
