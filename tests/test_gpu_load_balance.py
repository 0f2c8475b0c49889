"""The load-balance build (libmoira_cta_times.so) next to libmoira.so.

Both builds can be loaded in one process and used in either order: each
keeps its own record of the kernels' shared-memory limits (a record shared
between them made the second one's launches fail).  The timing build gives
the same outputs as libmoira.so bit for bit and a (start, end) pair for every
attention block that holds pages.
"""
import numpy as np
import pytest
import torch

import sparse_long_context_page_gb300 as moira
from sparse_long_context_page_gb300 import _binding as mb
from sparse_long_context_page_gb300 import build as B
from sparse_long_context_page_gb300 import workloads as W
from sparse_long_context_page_gb300.state import DecodeState

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _timed_step(st, gamma):
    nb = mb.attend_grid_blocks()
    buf = torch.zeros((st.layers, nb, 2), dtype=torch.int64, device="cuda")
    with mb.library_variant(B.LIB_CTA_TIMES):
        mb.set_cta_times(buf, st.layers)
        st.step(gamma)
        torch.cuda.synchronize()
        mb.set_cta_times(None, 0)
    return buf.cpu().numpy()


@pytest.mark.parametrize("name,over,timed_first", [
    ("llama8b_128k", dict(layers=2), False),           # few lists: 8
    ("serving_ragged", dict(batch=9, layers=2), True),  # many lists: 72
])
def test_timing_build_matches_and_records_every_block(name, over, timed_first):
    w = W.make_workload(name, seed=5, device="cuda", **over)
    st = DecodeState(w)
    st.summarize()
    g = float(np.float32(0.99))
    if timed_first:
        t = _timed_step(st, g)
        out_t, len_t = st.out.clone(), st.lengths.clone()
        st.step(g)
        torch.cuda.synchronize()
        out_m, len_m = st.out.clone(), st.lengths.clone()
    else:
        st.step(g)
        torch.cuda.synchronize()
        out_m, len_m = st.out.clone(), st.lengths.clone()
        t = _timed_step(st, g)
        out_t, len_t = st.out.clone(), st.lengths.clone()
    assert st.device_status() == 0
    assert torch.equal(len_t, len_m)
    assert torch.equal(out_t, out_m)
    nb = mb.attend_grid_blocks()
    for l in range(w.spec.layers):
        W_l = int(st.lengths[l].sum())
        s, e = t[l, :, 0], t[l, :, 1]
        busy = s > 0
        assert int(busy.sum()) == min(nb, W_l), (l, int(busy.sum()), W_l)
        assert np.all(e[busy] > s[busy])
        assert np.all((s[~busy] == 0) & (e[~busy] == 0))
        span = (e[busy].max() - s[busy].min()) / 1e3
        assert 1.0 < span < 10000.0, span                  # microseconds
