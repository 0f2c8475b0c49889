"""Contexts past 128k tokens, up to MAX_PAGES_PER_SEQ = 16384 pages (256k
tokens per request), against the fp64 oracle through the C ABI: the
selection's 16-stripe instantiation (two chunks per normaliser thread), the
score kernel over 512 chunks per request (single-wave and persistent launch
shapes), and attention over lists of several thousand pages."""
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


def _check(w, st, fmt, rules):
    G = w.group
    units = [(r, j) for r in range(w.spec.batch) for j in range(w.spec.kv_heads)]
    uds = {u: H.UnitData(w, 0, u[0], u[1], fmt=fmt) for u in units}
    for rule, param in rules:
        lists = torch.full_like(st.lists, -7)
        lengths = torch.zeros((w.spec.batch, w.spec.kv_heads), dtype=torch.int32, device="cuda")
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
            why = (H.check_list(ud, gl, param) if rule == mb.RULE_COVERAGE
                   else H.check_rule_list(ud, gl, rule, param))
            assert why is None, f"rule {rule} param {param} r{r} j{j} (L={ud.L}): {why}"
            ma, rl = H.out_errors(oh[r, j * G:(j + 1) * G], ud.attend(ud.to_logical(gl)))
            assert ma <= H.MAX_ABS and rl <= H.REL_L2, f"rule {rule} r{r} j{j}: {ma:.3g} {rl:.3g}"


RULES = ((mb.RULE_COVERAGE, float(np.float32(0.99))), (mb.RULE_COVERAGE, float(np.float32(0.9))),
         (mb.RULE_TOPK, 3000.0), (mb.RULE_TOPDELTA, 1e-3))


@pytest.mark.parametrize("fmt", [mb.SUMM_BF16, mb.SUMM_Q8])
def test_256k_tokens_single_request(fmt):
    """16383 full pages and a partial tail: the largest context one request may have."""
    ctx = 16 * mb.MAX_PAGES_PER_SEQ - 5
    w = W.make_workload("llama8b_128k", seed=61, device="cuda", layers=1, context=(ctx,))
    assert w.max_pages == mb.MAX_PAGES_PER_SEQ
    st = DecodeState(w, fmt=fmt)
    st.summarize()
    _check(w, st, fmt, RULES)
    del st, w
    torch.cuda.empty_cache()


def test_ragged_batch_across_128k():
    """Requests of 200k, 9k and 140k tokens in one call: 16 stripes in the
    selection and the persistent score walk (2 x 3 x 391 possible items)."""
    w = W.make_workload("llama8b_128k", seed=62, device="cuda", layers=1, batch=3,
                        context=(200000, 9000, 140001))
    st = DecodeState(w)
    st.summarize()
    _check(w, st, mb.SUMM_BF16, RULES[:1] + RULES[2:])
    del st, w
    torch.cuda.empty_cache()
