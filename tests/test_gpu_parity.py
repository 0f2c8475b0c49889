"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Inputs are the seeded synthetic workloads; sizes here keep the oracle at
seconds while spanning many score chunks, many attention blocks, ragged
tails and every selection regime.  Comparison rules: see helpers.py.
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


def _check_layer(w, st, l, gamma, units=None, check_out=True, stats=None):
    """Select + attend one layer on the GPU and compare every (or the given)
    unit with the oracle: its list by the comparison rules, and its output
    with the oracle's attention over the GPU's own list (so a list that
    differs at the gamma boundary is still checked).  Returns (units
    checked, outputs compared)."""
    lists = torch.zeros_like(st.lists)
    lengths = torch.zeros((w.spec.batch, w.spec.kv_heads), dtype=torch.int32, device="cuda")
    st.select_layer(l, gamma, lists, lengths)
    out = torch.zeros_like(st.out[l])
    st.attend_layer(l, lists, lengths, out)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    lists_h, len_h, out_h = lists.cpu().numpy(), lengths.cpu().numpy(), out.cpu().numpy()
    G = w.group
    units = units or [(r, j) for r in range(w.spec.batch) for j in range(w.spec.kv_heads)]
    n_out = 0
    for (r, j) in units:
        ud = H.UnitData(w, l, r, j)
        gl = lists_h[r, j, :len_h[r, j]]
        why = H.check_list(ud, gl, gamma, stats)
        assert why is None, f"layer {l} req {r} kv {j} gamma {gamma}: {why}"
        if check_out:
            lg = ud.to_logical(gl)
            if len(lg) == 0:
                assert np.all(out_h[r, j * G:(j + 1) * G] == 0.0), f"l{l} r{r} j{j}: empty list not zero"
            else:
                ma, rl = H.out_errors(out_h[r, j * G:(j + 1) * G], ud.attend(lg))
                assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"l{l} r{r} j{j}: max-abs {ma:.3g} rel-L2 {rl:.3g}"
            n_out += 1
    return len(units), n_out


# ------------------------------------------------------------------ summaries

def test_summaries_bit_exact():
    w, st = _state("llama8b_128k", seed=3, layers=2, context=(16 * 700 + 9,))
    torch.cuda.synchronize()
    got = H.u16(st.summ)                                           # [L][P][Hkv][d]
    k = H.u16(w.k_pool)                                            # [L][P][Hkv][S][d]
    ref = H.oracle.summaries(k.reshape(-1, 16, 128)).reshape(got.shape)
    diff = np.count_nonzero(got != ref)
    assert diff == 0, f"{diff} of {got.size} summary elements differ"


# ------------------------------------------------------------------ selection + attention

@pytest.mark.parametrize("gamma", [0.9, 0.99, 1.0])
def test_tiny_select_and_attend(gamma):
    w, st = _state("tiny", seed=0)
    n_units, n_out = _check_layer(w, st, 0, float(np.float32(gamma)))
    assert n_out == n_units


@pytest.mark.parametrize("name,over,gamma", [
    ("llama8b_32k", dict(layers=2), 0.99),
    ("llama8b_128k", dict(layers=1), 0.98),
    ("llama8b_128k", dict(layers=1), 0.99),
    ("serving_ragged", dict(batch=4, layers=1), 0.99),
    ("stress_regimes", dict(batch=6, context=(16 * 4000 + 7,)), 0.99),
])
def test_config_select_and_attend(name, over, gamma):
    w, st = _state(name, seed=11, **over)
    stats = {}
    for l in range(w.spec.layers):
        nu, no = _check_layer(w, st, l, float(np.float32(gamma)), stats=stats)
        assert no == nu
    assert stats.get("tie_only", 0) <= H.TIE_ONLY_MAX, stats


def test_select_edge_lengths():
    """Empty, sub-page, exact-page and tail-only contexts in one ragged batch,
    with max_pages larger than any request needs; gamma from one page (1e-6)
    to just below 1 (0.99999: the cut falls in the flat tail of masses far
    below the comparison band) and dense."""
    sp = W.spec("llama8b_128k", batch=8, layers=1, context=(0, 1, 15, 16, 17, 16 * 33, 16 * 257 + 3, 16 * 5000))
    w = W.make_workload(sp, seed=5, device="cuda")
    st = DecodeState(w, max_pages=w.max_pages + 37)
    st.summarize()
    for gamma in (1e-6, 0.5, 0.99, 0.99999, 1.0):
        _check_layer(w, st, 0, float(np.float32(gamma)))


@pytest.mark.parametrize("batch", [5, 8, 12])
def test_attend_random_lists_isolated(batch):
    """Attention alone on seeded random lists (neither side's selection).
    40 lists run the attention kernel's small-batch shape (4 consumer warps,
    12-slot ring); 64 (the switch-over) and 96 run the many-list shape (5
    consumer warps, 10-slot ring), long lists included."""
    w = W.make_workload("serving_ragged", seed=21, device="cuda", batch=batch, layers=1)
    st = DecodeState(w)
    G = w.group
    for trial, frac in enumerate([(0.0, 1.0), (0.0, 0.02), (0.9, 1.0)]):
        logical, phys, lengths = W.random_lists(w, seed=100 + trial, keep_frac=frac)
        lists = torch.from_numpy(phys).cuda()
        lens = torch.from_numpy(lengths).cuda()
        out = torch.zeros_like(st.out[0])
        st.attend_layer(0, lists, lens, out)
        torch.cuda.synchronize()
        assert st.device_status() == 0
        oh = out.cpu().numpy()
        for r in range(w.spec.batch):
            for j in range(w.spec.kv_heads):
                ud = H.UnitData(w, 0, r, j)
                ref = ud.attend(logical[r][j])
                ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ref)
                assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"{frac} r{r} j{j}: {ma:.3g} {rl:.3g}"


@pytest.mark.parametrize("batch", [3, 32])
def test_attend_empty_and_single_lists(batch):
    """Empty lists give zeros; one full page, the tail page alone and a whole
    context give the oracle's attention.  Every list keeps the contract: a
    request's partial tail page, when it has one and the list is not empty,
    is the list's last entry.  3 requests (6 lists) run the attention
    kernel's small-batch shape, 32 requests (64 lists) its many-list shape."""
    ctx = tuple(16 * 40 + (3 if r % 3 == 1 else 0) for r in range(batch))
    w = W.make_workload("tiny", seed=2, device="cuda", batch=batch, context=ctx)
    st = DecodeState(w)
    B, Hkv = batch, w.spec.kv_heads
    phys = np.full((B, Hkv, w.max_pages), -1, np.int32)
    lengths = np.zeros((B, Hkv), np.int32)
    logical = [[np.zeros(0, np.int32) for _ in range(Hkv)] for _ in range(B)]
    for r in range(B):
        F, T = ctx[r] // 16, int(ctx[r] % 16 != 0)
        for j in range(Hkv):
            kind = (r * Hkv + j) % 4
            if kind == 1:      # one full page, and the tail, which the contract puts last
                logical[r][j] = np.array([7, F] if T else [7], np.int32)
            elif kind == 2:    # the tail page alone (3 tokens), or the last full page
                logical[r][j] = np.array([F if T else F - 1], np.int32)
            elif kind == 3:    # everything
                logical[r][j] = np.arange(F + T, dtype=np.int32)
            lst = logical[r][j]
            phys[r, j, :len(lst)] = w.page_table[r, lst]
            lengths[r, j] = len(lst)
    out = torch.full_like(st.out[0], 7.0)
    st.attend_layer(0, torch.from_numpy(phys).cuda(), torch.from_numpy(lengths).cuda(), out)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    oh = out.cpu().numpy()
    G = w.group
    for r in range(B):
        for j in range(Hkv):
            if len(logical[r][j]) == 0:
                assert np.all(oh[r, j * G:(j + 1) * G] == 0.0), f"r{r} j{j}: empty list not zero"
                continue
            ref = H.UnitData(w, 0, r, j).attend(logical[r][j])
            ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ref)
            assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"r{r} j{j}: {ma:.3g} {rl:.3g}"


# ------------------------------------------------------------------ graph, status, determinism

def test_graph_capture_matches_eager_bit_for_bit():
    w, st = _state("llama8b_32k", seed=4, layers=4)
    st.step(0.99)
    torch.cuda.synchronize()
    out_e, len_e = st.out.clone(), st.lengths.clone()
    st.out.zero_()
    st.lengths.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st.step(0.99)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.lengths, len_e)
    assert torch.equal(st.out, out_e)
    assert st.device_status() == 0


def test_device_status_flags_bad_pages_and_lengths():
    w, st = _state("tiny", seed=6)
    pt = st.page_table.clone()
    st.page_table[0, 3] = w.num_phys_pages + 5                     # out of the pool
    lists, lengths = st.select_layer(0, 0.99)
    out = st.attend_layer(0, lists, lengths)
    torch.cuda.synchronize()
    assert st.device_status() & mb.DEV_BADPAGE
    st.page_table.copy_(pt)
    bad_len = torch.full_like(st.lengths[0], st.max_pages + 100)
    st.attend_layer(0, st.lists, bad_len)
    torch.cuda.synchronize()
    assert st.device_status() & mb.DEV_BADLEN
    # the context is still usable and clean afterwards
    st.step(0.99)
    torch.cuda.synchronize()
    assert st.device_status() == 0


def test_host_checks_launch_nothing():
    w, st = _state("tiny", seed=7)
    with pytest.raises(mb.MoiraError):
        st.select_layer(0, 1.5)
    with pytest.raises(mb.MoiraError):
        st.select_layer(0, 0.0)
    small = st.ws[: st.ws.numel() // 2]
    with pytest.raises(mb.MoiraError):
        mb.select(st.shape, w.q[0], st.summ[0], st.page_table, st.seq_lens, 0.9, st.sm_scale,
                  st.lists, st.lengths[0], small)


def test_host_buffers_step_matches_device_step():
    w, st = _state("llama8b_32k", seed=8, layers=2)
    st.step(0.99)
    torch.cuda.synchronize()
    ref = st.out.clone()
    q_host = w.q.cpu().pin_memory()
    out_host = torch.empty(st.out.shape, dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(w.q)
    out_dev = torch.empty_like(st.out)
    mb.decode_step_host(st.shape, q_host, q_dev, w.k_pool, w.v_pool, st.summ, st.page_table,
                        st.seq_lens, 0.99, st.sm_scale, st.lists, st.lengths, out_dev, out_host, st.ws)
    torch.cuda.synchronize()
    assert torch.equal(out_host, ref.cpu())


@pytest.mark.parametrize("fmt", [mb.SUMM_BF16, mb.SUMM_Q8])
@pytest.mark.parametrize("persistent", [False, True])
def test_decode_step_matches_per_layer_calls(fmt, persistent):
    """From layer 1 on, the decode step lets the score kernel read the page
    table and the lengths before its dependency wait; the per-layer calls
    (moira_select_attend, and moira_select for the lists) wait first.  Both
    must give the same lengths, lists and outputs, bit for bit, under both
    launch shapes of the score kernel (one request takes the single-launch
    selection + attention, three requests of 8192 pages the two-launch form)."""
    if persistent:
        over = dict(batch=3, context=(16 * 700 + 9, 16 * 1500 + 3, 16 * 300))
        max_pages = 8192                   # 3 x 2 x 256 items: more than one wave
    else:
        over = dict(batch=1, context=(16 * 900 + 5,))
        max_pages = None
    w = W.make_workload("llama8b_32k", seed=50, device="cuda", layers=4, **over)
    st = DecodeState(w, max_pages=max_pages, fmt=fmt)
    st.summarize()
    gamma = float(np.float32(0.99))
    st.step(gamma)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    out_s, len_s, last_lists = st.out.clone(), st.lengths.clone(), st.lists.clone()
    for l in range(w.spec.layers):
        lists = torch.full_like(st.lists, -1)
        lengths = torch.zeros_like(st.lengths[l])
        out = torch.zeros_like(st.out[l])
        st.select_attend_layer(l, gamma, lists, lengths, out)
        sel_lists = torch.full_like(st.lists, -1)
        sel_len = torch.zeros_like(st.lengths[l])
        st.select_layer(l, gamma, sel_lists, sel_len)
        torch.cuda.synchronize()
        assert torch.equal(lengths, len_s[l]), f"layer {l}: list lengths differ"
        assert torch.equal(sel_len, len_s[l]), f"layer {l}: moira_select's lengths differ"
        assert torch.equal(out, out_s[l]), f"layer {l}: outputs differ"
    n = lengths.cpu().numpy()
    lh, ls, sh = lists.cpu().numpy(), last_lists.cpu().numpy(), sel_lists.cpu().numpy()
    for r in range(w.spec.batch):
        for j in range(w.spec.kv_heads):
            assert np.array_equal(lh[r, j, :n[r, j]], ls[r, j, :n[r, j]])
            assert np.array_equal(sh[r, j, :n[r, j]], ls[r, j, :n[r, j]])
    assert st.device_status() == 0


# ------------------------------------------------------------------ full sizes, sampled units

FULL = [("llama8b_32k", 0.99), ("llama8b_128k", 0.99), ("llama8b_128k", 0.98),
        ("stress_regimes", 0.99), ("serving_ragged", 0.99)]


@pytest.mark.parametrize("name,gamma", FULL)
def test_full_size_sampled_units(name, gamma):
    """The full configuration, whole step in one graph (as the benchmark runs
    it); sampled units are checked against the oracle one by one."""
    torch.cuda.empty_cache()
    w, st = _state(name, seed=0)
    g32 = float(np.float32(gamma))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        st.step(g32)                                               # warm-up (sets attributes)
        with torch.cuda.graph(g, stream=s):
            st.step(g32)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert st.device_status() == 0
    rng = np.random.default_rng(123)
    L, B, Hkv, G = w.spec.layers, w.spec.batch, w.spec.kv_heads, w.group
    picks = sorted({(int(rng.integers(L)), int(rng.integers(B)), int(rng.integers(Hkv))) for _ in range(48)})
    out_h = st.out.cpu().numpy()
    len_h = st.lengths.cpu().numpy()
    lists = torch.zeros_like(st.lists)
    stats = {}
    for l in sorted({p[0] for p in picks}):
        lengths = torch.zeros((B, Hkv), dtype=torch.int32, device="cuda")
        st.select_layer(l, g32, lists, lengths)        # the step keeps only the last layer's lists
        torch.cuda.synchronize()
        lh, ph = lengths.cpu().numpy(), lists.cpu().numpy()
        assert np.array_equal(lh, len_h[l])
        for (_, r, j) in [p for p in picks if p[0] == l]:
            gl = ph[r, j, :lh[r, j]]
            ud = H.UnitData(w, l, r, j)
            why = H.check_list(ud, gl, g32, stats)
            assert why is None, f"{name} l{l} r{r} j{j}: {why}"
            ma, rl = H.out_errors(out_h[l, r, j * G:(j + 1) * G], ud.attend(ud.to_logical(gl)))
            assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"{name} l{l} r{r} j{j}: {ma:.3g} {rl:.3g}"
    assert stats.get("tie_only", 0) <= H.TIE_ONLY_MAX, stats
    del st, w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("F", [50, 500, 3000])
def test_select_all_masses_tied(F):
    """Identical keys give identical masses: the rule keeps the ceil(gamma*F)
    lowest logical pages (plus the tail).  F = 50, 500 and 3000 take the
    pairwise, single-warp and block-wide refinement paths respectively."""
    L = 16 * F + 5
    sp = W.spec("llama8b_128k", batch=1, layers=1, context=(L,))
    w = W.make_workload(sp, seed=9, device="cuda")
    key = torch.randn(128, generator=torch.Generator(device="cuda").manual_seed(1), device="cuda")
    w.k_pool[:] = key.to(torch.bfloat16)
    st = DecodeState(w)
    st.summarize()
    for gamma in (0.3, 0.7, 0.9, 0.99):
        g = float(np.float32(gamma))
        k = int(np.ceil(g * F))
        lists, lengths = st.select_layer(0, g)
        torch.cuda.synchronize()
        assert st.device_status() == 0
        lh, nh = lists.cpu().numpy(), lengths.cpu().numpy()
        for j in range(w.spec.kv_heads):
            ud = H.UnitData(w, 0, 0, j, with_v=False)
            why = H.check_list(ud, lh[0, j, :nh[0, j]], g)
            assert why is None, f"F={F} gamma={g} head {j}: {why}"
            logical = ud.to_logical(lh[0, j, :nh[0, j]])
            if abs(g * F - round(g * F)) > 1e-3:           # away from an integer: exact
                assert list(logical) == list(range(k)) + [F], f"F={F} gamma={g}: {len(logical)} vs {k}+1"


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("llama8b_32k", dict(layers=1)),
    ("serving_ragged", dict(batch=3, layers=1)),
    ("stress_regimes", dict(batch=4, context=(16 * 2000 + 9,))),
])
def test_select_rules_topk_and_topdelta(name, over):
    """Fixed-budget and relative-threshold rules through the same kernels:
    lists against the oracle rules on the oracle masses, and attention over
    the GPU's own lists against the oracle's attention."""
    w, st = _state(name, seed=29, **over)
    G = w.group
    cases = [(mb.RULE_TOPK, 0), (mb.RULE_TOPK, 1), (mb.RULE_TOPK, 37), (mb.RULE_TOPK, 600),
             (mb.RULE_TOPK, 1 << 20), (mb.RULE_TOPDELTA, 1.0), (mb.RULE_TOPDELTA, 0.3),
             (mb.RULE_TOPDELTA, 1e-3)]
    units = [(r, j) for r in range(w.spec.batch) for j in range(w.spec.kv_heads)]
    uds = {u: H.UnitData(w, 0, u[0], u[1]) for u in units}
    for rule, param in cases:
        lists = torch.full_like(st.lists, -7)
        lengths = torch.zeros((w.spec.batch, w.spec.kv_heads), dtype=torch.int32, device="cuda")
        st.select_layer_rule(0, rule, float(param), lists, lengths)
        out = torch.zeros_like(st.out[0])
        st.attend_layer(0, lists, lengths, out)
        torch.cuda.synchronize()
        assert st.device_status() == 0, (name, rule, param)
        lh, nh, oh = lists.cpu().numpy(), lengths.cpu().numpy(), out.cpu().numpy()
        for (r, j) in units:
            ud = uds[(r, j)]
            gl = lh[r, j, :nh[r, j]]
            why = H.check_rule_list(ud, gl, rule, float(param))
            assert why is None, f"{name} rule {rule} param {param} req {r} kv {j}: {why}"
            lg = ud.to_logical(gl)
            if len(lg):
                ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ud.attend(lg))
                assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"{name} {rule}/{param} r{r} j{j}: {ma:.3g} {rl:.3g}"
    del st, w
    torch.cuda.empty_cache()


def test_select_rule_coverage_is_select_bit_for_bit():
    w, st = _state("serving_ragged", seed=31, batch=3, layers=1)
    for g in (0.5, 0.9, 0.99):
        g = float(np.float32(g))
        a_l, a_n = torch.full_like(st.lists, -7), torch.zeros_like(st.lengths[0])
        b_l, b_n = torch.full_like(st.lists, -7), torch.zeros_like(st.lengths[0])
        st.select_layer(0, g, a_l, a_n)
        st.select_layer_rule(0, mb.RULE_COVERAGE, g, b_l, b_n)
        torch.cuda.synchronize()
        assert torch.equal(a_n, b_n)
        for r in range(w.spec.batch):
            for j in range(w.spec.kv_heads):
                n = int(a_n[r, j])
                assert torch.equal(a_l[r, j, :n], b_l[r, j, :n])


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    """The bounded device wait, made to run out on purpose (an mbarrier that
    nothing completes, 50 ms limit): MOIRA_DEV_TIMEOUT reaches the host through
    the status word, and the same workspace then serves a normal step."""
    import time
    w, st = _state("tiny", seed=0)
    assert st.device_status() == 0
    t0 = time.perf_counter()
    mb.diag_wait_timeout(st.ws, 50_000_000)
    status = mb.read_device_status(st.ws)                 # synchronises, clears
    took = time.perf_counter() - t0
    assert status & mb.DEV_TIMEOUT, hex(status)
    assert 0.04 < took < 5.0, took
    _check_layer(w, st, 0, float(np.float32(0.9)))        # select + attend still correct
    assert st.device_status() == 0


def test_maximum_unit_count():
    """4096 (request, KV head) units, the most one call takes: 512 requests of
    1-400 tokens (ragged, with tails and with requests shorter than a page).
    Every list is well formed and kept within its request; a sample of units
    is checked against the oracle, lists and outputs."""
    rng = np.random.default_rng(77)
    ctx = tuple(int(x) for x in rng.integers(1, 400, size=512))
    w, st = _state("llama8b_32k", seed=77, layers=1, batch=512, context=ctx)
    assert w.spec.batch * w.spec.kv_heads == mb.MAX_UNITS
    g = float(np.float32(0.9))
    lists = torch.full_like(st.lists, -7)
    lengths = torch.zeros((w.spec.batch, w.spec.kv_heads), dtype=torch.int32, device="cuda")
    st.select_layer(0, g, lists, lengths)
    out = torch.zeros_like(st.out[0])
    st.attend_layer(0, lists, lengths, out)
    torch.cuda.synchronize()
    assert st.device_status() == 0
    lh, nh, oh = lists.cpu().numpy(), lengths.cpu().numpy(), out.cpu().numpy()
    seq = w.seq_lens
    for r in range(w.spec.batch):
        n_pages = (int(seq[r]) + 15) // 16
        row = set(int(p) for p in w.page_table[r, :n_pages])
        for j in range(w.spec.kv_heads):
            n = int(nh[r, j])
            assert 1 <= n <= n_pages, (r, j, n, n_pages)
            assert set(int(p) for p in lh[r, j, :n]) <= row
            if seq[r] % 16:
                assert lh[r, j, n - 1] == w.page_table[r, n_pages - 1]
    G = w.group
    for _ in range(48):
        r, j = int(rng.integers(w.spec.batch)), int(rng.integers(w.spec.kv_heads))
        ud = H.UnitData(w, 0, r, j)
        gl = lh[r, j, :nh[r, j]]
        why = H.check_list(ud, gl, g)
        assert why is None, f"r{r} j{j}: {why}"
        ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ud.attend(ud.to_logical(gl)))
        assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"r{r} j{j}: {ma:.3g} {rl:.3g}"
