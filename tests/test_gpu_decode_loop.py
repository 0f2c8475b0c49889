"""A decode loop: every step appends one token per request to every layer
(moira_append_kv, which writes a page's summary when the page fills) and then
runs the decode step, all in order on one stream.

Inside the step, the scoring kernels of layers 1 and later read the page
table and start their summary copies before their dependency wait (the
kernel before them is the previous layer's attention, which writes neither);
the step's first scoring launch waits for everything the caller queued,
the appends included.  The loop must therefore give exactly what the same
loop gives with the device synchronised between every append and step, and
its last step must match the oracle.
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

# the last page of each request is partial: 8 and 7 free slots, so eight appends
# fill the first request's page (its summary is written by the append of step 8)
CONTEXT = (16 * 300 + 8, 16 * 123 + 7)
STEPS = 8


def _loop(sync: bool):
    sp = W.spec("llama8b_32k", batch=2, layers=4, context=CONTEXT)
    w = W.make_workload(sp, seed=77, device="cuda")
    st = DecodeState(w)
    st.summarize()
    B, Hkv, L = sp.batch, sp.kv_heads, sp.layers
    gen = torch.Generator(device="cuda").manual_seed(5)
    outs, lens, lists = [], [], []
    g32 = float(np.float32(0.99))
    for _ in range(STEPS):
        st.seq_lens += 1
        for l in range(L):
            k_new = torch.randn((B, Hkv, 128), generator=gen, device="cuda").to(torch.bfloat16)
            v_new = torch.randn((B, Hkv, 128), generator=gen, device="cuda").to(torch.bfloat16)
            mb.append_kv(st.shape, k_new, v_new, w.k_pool[l], w.v_pool[l], st.summ[l], st.page_table,
                         st.seq_lens)
        if sync:
            torch.cuda.synchronize()
        st.step(g32)
        outs.append(st.out.clone())
        lens.append(st.lengths.clone())
        lists.append(st.lists.clone())
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    assert st.device_status() == 0
    return w, st, outs, lens, lists


def test_decode_loop_with_appends_is_ordered():
    _, _, outs_a, lens_a, lists_a = _loop(sync=False)
    w, st, outs_b, lens_b, lists_b = _loop(sync=True)
    for s in range(STEPS):
        assert torch.equal(lens_a[s], lens_b[s]), f"step {s}: lengths differ"
        assert torch.equal(outs_a[s], outs_b[s]), f"step {s}: outputs differ"
        n = lens_b[s][-1].cpu().numpy()                      # the last layer's lists are kept
        la, lb = lists_a[s].cpu().numpy(), lists_b[s].cpu().numpy()
        for r in range(w.spec.batch):
            for j in range(w.spec.kv_heads):
                assert np.array_equal(la[r, j, :n[r, j]], lb[r, j, :n[r, j]]), f"step {s} list ({r},{j})"
    # the last step against the oracle, last layer (the appended tokens included)
    assert int(st.seq_lens[0]) == CONTEXT[0] + STEPS and (CONTEXT[0] + STEPS) % 16 == 0
    l = w.spec.layers - 1
    lh, nh, oh = lists_b[-1].cpu().numpy(), lens_b[-1][l].cpu().numpy(), outs_b[-1][l].cpu().numpy()
    w.seq_lens[:] = st.seq_lens.cpu().numpy()
    G = w.group
    for r in range(w.spec.batch):
        for j in range(w.spec.kv_heads):
            ud = H.UnitData(w, l, r, j)
            gl = lh[r, j, :nh[r, j]]
            why = H.check_list(ud, gl, float(np.float32(0.99)))
            assert why is None, f"req {r} kv {j}: {why}"
            ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ud.attend(ud.to_logical(gl)))
            assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"req {r} kv {j}: {ma:.3g} {rl:.3g}"
