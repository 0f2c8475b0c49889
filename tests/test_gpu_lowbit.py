"""Parity of the low-bit page-summary path (8-bit and 2-bit mid-rise mean keys)
with the fp64 oracle, through the C ABI.

Summaries are integer work (codes) plus one fp32 step decided in fp64 on
both sides, so they must match the oracle's records bit for bit.  Lists and
outputs follow the comparison rules of helpers.py with the oracle's masses
taken from the oracle's own low-bit summaries.
"""
import numpy as np
import pytest
import torch

import helpers as H
from oracle import oracle
import sparse_long_context_page_gb300 as moira
from sparse_long_context_page_gb300 import _binding as mb
from sparse_long_context_page_gb300 import workloads as W
from sparse_long_context_page_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

D, S = 128, 16
FMTS = [(mb.SUMM_Q8, 8), (mb.SUMM_Q2, 2)]


def _state(name, fmt, seed=0, **over):
    w = W.make_workload(name, seed=seed, device="cuda", **over)
    st = DecodeState(w, fmt=fmt)
    st.summarize()
    return w, st


def _oracle_records(k_pool_layer, bits, rec_bytes):
    """The oracle's low-bit summaries of a whole layer pool, as records."""
    k = H.u16(k_pool_layer)                                         # [P][Hkv][S][d]
    P, Hkv = k.shape[:2]
    codes, steps = oracle.summaries_lowbit(k.reshape(-1, S, D), bits)
    return H.pack_lowbit(codes.reshape(P, Hkv, D), steps.reshape(P, Hkv), bits, rec_bytes)


@pytest.mark.parametrize("fmt,bits", FMTS)
def test_lowbit_summaries_bit_exact(fmt, bits):
    """Every record of two layers, with degenerate pages planted in layer 0:
    all-zero keys, an infinite key, a NaN key, a lone subnormal (the step is
    then an fp32 subnormal and the top code is clamped), and huge keys."""
    w = W.make_workload("llama8b_128k", seed=3, device="cuda", layers=2, context=(16 * 700 + 9,))
    st = DecodeState(w, fmt=fmt)
    kp = w.k_pool[0]
    kp[1].zero_()
    kp[2, 0, 5, 7] = float("inf")
    kp[3, 1, 0, 0] = float("nan")
    kp[4].zero_()
    kp[4].view(torch.int16)[0, 3, 9] = 0x0001                       # smallest bf16 subnormal
    kp[5, 1].view(torch.int16)[2, 11] = -0x7FFF                     # bit pattern 0x8001: -2^-133
    kp[6] *= 1e30
    st.summarize()
    torch.cuda.synchronize()
    rec = mb.summary_page_bytes(st.shape, fmt)
    assert st.summ.shape == (2, w.num_phys_pages, rec)
    for l in range(2):
        got = st.summ[l].cpu().numpy()
        want = _oracle_records(w.k_pool[l], bits, rec)
        bad = np.argwhere(got != want)
        assert bad.size == 0, f"layer {l}: {len(bad)} bytes differ, first at (page, byte) {bad[:4].tolist()}"


def _check_units(w, st, l, gamma, fmt, lists, lengths, out):
    lh, nh, oh = lists.cpu().numpy(), lengths.cpu().numpy(), out.cpu().numpy()
    G = w.group
    n_out = 0
    for r in range(w.spec.batch):
        for j in range(w.spec.kv_heads):
            ud = H.UnitData(w, l, r, j, fmt=fmt)
            gl = lh[r, j, :nh[r, j]]
            why = H.check_list(ud, gl, gamma)
            assert why is None, f"fmt {fmt} layer {l} req {r} kv {j} gamma {gamma}: {why}"
            o_list = ud.select(gamma)[0]
            if np.array_equal(ud.to_logical(gl), o_list):
                ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ud.attend(o_list))
                assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"fmt {fmt} l{l} r{r} j{j}: {ma:.3g} {rl:.3g}"
                n_out += 1
    return n_out


@pytest.mark.parametrize("fmt,bits", FMTS)
@pytest.mark.parametrize("name,over,gammas", [
    ("tiny", {}, (0.9, 0.99, 1.0)),
    ("llama8b_32k", dict(layers=1), (0.99,)),
    ("serving_ragged", dict(batch=3, layers=1), (0.99,)),
    ("stress_regimes", dict(batch=4, context=(16 * 2000 + 9,)), (0.99,)),
])
def test_lowbit_select_and_attend(fmt, bits, name, over, gammas):
    w, st = _state(name, fmt, seed=17, **over)
    units = w.spec.batch * w.spec.kv_heads
    for gamma in gammas:
        g32 = float(np.float32(gamma))
        lists = torch.full_like(st.lists, -7)
        lengths = torch.zeros((w.spec.batch, w.spec.kv_heads), dtype=torch.int32, device="cuda")
        st.select_layer(0, g32, lists, lengths)
        out = torch.zeros_like(st.out[0])
        st.attend_layer(0, lists, lengths, out)
        torch.cuda.synchronize()
        assert st.device_status() == 0
        n_out = _check_units(w, st, 0, g32, fmt, lists, lengths, out)
        assert n_out >= units - 2, (name, gamma, n_out, units)
    del st, w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt,bits", FMTS)
def test_lowbit_rules(fmt, bits):
    """Top-k and top-delta read the same low-bit estimate."""
    w, st = _state("stress_regimes", fmt, seed=23, batch=4, context=(16 * 2000 + 9,))
    units = [(r, j) for r in range(w.spec.batch) for j in range(w.spec.kv_heads)]
    uds = {u: H.UnitData(w, 0, u[0], u[1], fmt=fmt) for u in units}
    for rule, param in [(mb.RULE_TOPK, 0), (mb.RULE_TOPK, 37), (mb.RULE_TOPK, 1 << 20),
                        (mb.RULE_TOPDELTA, 1.0), (mb.RULE_TOPDELTA, 1e-2)]:
        lists = torch.full_like(st.lists, -7)
        lengths = torch.zeros((w.spec.batch, w.spec.kv_heads), dtype=torch.int32, device="cuda")
        st.select_layer_rule(0, rule, float(param), lists, lengths)
        torch.cuda.synchronize()
        assert st.device_status() == 0
        lh, nh = lists.cpu().numpy(), lengths.cpu().numpy()
        for (r, j) in units:
            why = H.check_rule_list(uds[(r, j)], lh[r, j, :nh[r, j]], rule, float(param))
            assert why is None, f"fmt {fmt} rule {rule} param {param} r{r} j{j}: {why}"


@pytest.mark.parametrize("fmt,bits", FMTS)
def test_lowbit_step_graph_matches_eager_and_oracle(fmt, bits):
    """moira_decode_step_ex over four layers: a graph replay equals the eager
    call bit for bit, and every unit of two layers passes the oracle check."""
    w, st = _state("llama8b_32k", fmt, seed=4, layers=4)
    g32 = float(np.float32(0.99))
    st.step(g32)
    torch.cuda.synchronize()
    len_e, out_e = st.lengths.clone(), st.out.clone()
    st.lengths.zero_()
    st.out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st.step(g32)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert st.device_status() == 0
    assert torch.equal(st.lengths, len_e) and torch.equal(st.out, out_e)
    for l in (0, 3):
        lists = torch.zeros_like(st.lists)
        lengths = torch.zeros_like(st.lengths[l])
        st.select_layer(l, g32, lists, lengths)
        torch.cuda.synchronize()
        assert torch.equal(lengths, st.lengths[l])
        _check_units(w, st, l, g32, fmt, lists, lengths, st.out[l])


@pytest.mark.parametrize("fmt,bits", FMTS)
def test_lowbit_full_size_sampled_units(fmt, bits):
    """The 128k configuration, whole 32-layer step in one graph, sampled
    units against the oracle."""
    torch.cuda.empty_cache()
    w, st = _state("llama8b_128k", fmt, seed=0)
    g32 = float(np.float32(0.99))
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        st.step(g32)
        with torch.cuda.graph(g, stream=s):
            st.step(g32)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert st.device_status() == 0
    rng = np.random.default_rng(321)
    L, Hkv, G = w.spec.layers, w.spec.kv_heads, w.group
    picks = sorted({(int(rng.integers(L)), int(rng.integers(Hkv))) for _ in range(6)})
    out_h, len_h = st.out.cpu().numpy(), st.lengths.cpu().numpy()
    lists = torch.zeros_like(st.lists)
    compared = 0
    for (l, j) in picks:
        lengths = torch.zeros((1, Hkv), dtype=torch.int32, device="cuda")
        st.select_layer(l, g32, lists, lengths)
        torch.cuda.synchronize()
        lh = lengths.cpu().numpy()
        assert lh[0, j] == len_h[l, 0, j]
        gl = lists[0, j, :lh[0, j]].cpu().numpy()
        ud = H.UnitData(w, l, 0, j, fmt=fmt)
        why = H.check_list(ud, gl, g32)
        assert why is None, f"fmt {fmt} l{l} j{j}: {why}"
        o_list = ud.select(g32)[0]
        if np.array_equal(ud.to_logical(gl), o_list):
            ma, rl = H.out_errors(out_h[l, 0, j * G:(j + 1) * G], ud.attend(o_list))
            assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"fmt {fmt} l{l} j{j}: {ma:.3g} {rl:.3g}"
            compared += 1
    assert compared >= len(picks) - 1
    del st, w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt,bits", FMTS)
def test_lowbit_append_decode_loop(fmt, bits):
    """Forty appends with low-bit summaries: every page that fills gets the
    oracle's record of the final pool, and no other record changes."""
    P, Hkv, B, max_pages = 96, 4, 3, 24
    shape = moira.Shape.of(4 * Hkv, Hkv, P)
    g = torch.Generator(device="cuda").manual_seed(5)
    k_pool = torch.randn((P, Hkv, S, D), generator=g, device="cuda").to(torch.bfloat16)
    v_pool = torch.randn((P, Hkv, S, D), generator=g, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(6)
    table = rng.permutation(P)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    lens = np.array([16 * 2 + 5, 16 * 7, 1], np.int32)
    rec = moira.summary_page_bytes(shape, fmt)
    summ = moira.make_summaries(shape, fmt)
    full0 = np.concatenate([table[r, :lens[r] // S] for r in range(B)]).astype(np.int32)
    moira.update_summaries(shape, k_pool, summ, torch.from_numpy(full0).cuda(), fmt=fmt)
    pt = torch.from_numpy(table).cuda()
    for step in range(40):
        lens = lens + 1
        k_new = torch.randn((B, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
        v_new = torch.randn((B, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
        moira.append_kv(shape, k_new, v_new, k_pool, v_pool, summ, pt, torch.from_numpy(lens).cuda(),
                        fmt=fmt)
    torch.cuda.synchronize()
    want = _oracle_records(k_pool, bits, rec)
    got = summ.cpu().numpy()
    full = {int(table[r, lp]) for r in range(B) for lp in range(lens[r] // S)}
    for p in range(P):
        if p in full:
            assert np.array_equal(got[p], want[p]), p
        else:
            assert not got[p].any(), p                                 # never summarised
