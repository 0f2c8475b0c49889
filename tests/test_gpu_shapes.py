"""Every supported KV-head count (Hkv = 1, 2, 4, 8 with the GQA group of 4)
under every page-summary format and both launch shapes of the score kernel
(one block per item when the items fit in one wave; the persistent
device-planned walk otherwise), against the fp64 oracle through the C ABI.

Hkv below 4 gives score items of fewer than 4 heads (idle consumer warps)
and low-bit head groups with padding after the steps; the persistent walk
is forced by a wide page table (8192 pages) over three requests of uneven
length, which leaves most items empty.
"""
import numpy as np
import pytest
import torch

import helpers as H
from oracle import oracle
from sparse_long_context_page_gb300 import _binding as mb
from sparse_long_context_page_gb300 import workloads as W
from sparse_long_context_page_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

D, S = 128, 16
BITS = {mb.SUMM_Q8: 8, mb.SUMM_Q2: 2}


@pytest.mark.parametrize("persistent", [False, True])
@pytest.mark.parametrize("fmt", [mb.SUMM_BF16, mb.SUMM_Q8, mb.SUMM_Q2])
@pytest.mark.parametrize("hkv", [1, 2, 4, 8])
def test_kv_head_counts_formats_and_launch_shapes(hkv, fmt, persistent):
    if persistent:
        over = dict(batch=3, context=(16 * 700 + 9, 16 * 1500 + 3, 16 * 300))
        max_pages = 8192                   # 3 x (Hkv / min(Hkv, 4)) x 256 items: more than one wave
    else:
        over = dict(batch=1, context=(16 * 900 + 5,))
        max_pages = None
    w = W.make_workload("llama8b_32k", seed=40 + hkv, device="cuda", layers=1, q_heads=4 * hkv,
                        kv_heads=hkv, **over)
    st = DecodeState(w, max_pages=max_pages, fmt=fmt)
    st.summarize()
    torch.cuda.synchronize()
    if fmt != mb.SUMM_BF16:
        bits = BITS[fmt]
        k = H.u16(w.k_pool[0])
        codes, steps = oracle.summaries_lowbit(k.reshape(-1, S, D), bits)
        P = k.shape[0]
        want = H.pack_lowbit(codes.reshape(P, hkv, D), steps.reshape(P, hkv), bits,
                             mb.summary_page_bytes(st.shape, fmt))
        assert np.array_equal(st.summ[0].cpu().numpy(), want)
    else:
        got = H.u16(st.summ[0])
        want = oracle.summaries(H.u16(w.k_pool[0]).reshape(-1, S, D)).reshape(got.shape)
        assert np.array_equal(got, want)
    G = w.group
    units = [(r, j) for r in range(w.spec.batch) for j in range(hkv)]
    uds = {u: H.UnitData(w, 0, u[0], u[1], fmt=fmt) for u in units}
    for rule, param in ((mb.RULE_COVERAGE, float(np.float32(0.99))), (mb.RULE_TOPK, 40.0)):
        lists = torch.full_like(st.lists, -7)
        lengths = torch.zeros((w.spec.batch, hkv), dtype=torch.int32, device="cuda")
        if rule == mb.RULE_COVERAGE:
            st.select_layer(0, param, lists, lengths)
        else:
            st.select_layer_rule(0, rule, param, lists, lengths)
        out = torch.zeros_like(st.out[0])
        st.attend_layer(0, lists, lengths, out)
        torch.cuda.synchronize()
        assert st.device_status() == 0
        lh, nh, oh = lists.cpu().numpy(), lengths.cpu().numpy(), out.cpu().numpy()
        for (r, j) in units:
            ud = uds[(r, j)]
            gl = lh[r, j, :nh[r, j]]
            if rule == mb.RULE_COVERAGE:
                why = H.check_list(ud, gl, param)
            else:
                why = H.check_rule_list(ud, gl, rule, param)
            assert why is None, f"Hkv {hkv} fmt {fmt} rule {rule} r{r} j{j}: {why}"
            lg = ud.to_logical(gl)
            ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ud.attend(lg))
            assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"Hkv {hkv} fmt {fmt} r{r} j{j}: {ma:.3g} {rl:.3g}"
    del st, w
    torch.cuda.empty_cache()
