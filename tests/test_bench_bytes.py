"""The benchmark's algorithmic bytes (the roofline numerator) against a case
counted by hand: per layer, the summaries of every full page (only when an
estimate runs, gamma < 1), K and V of the listed tokens with a partial tail
page counted at its valid tokens, q in (bf16) and out (fp32)."""
from types import SimpleNamespace

import numpy as np
import pytest

import bench


def _workload():
    spec = SimpleNamespace(batch=2, layers=1, q_heads=8, kv_heads=2, head_dim=128, page_size=16)
    # request 0: 40 tokens = 2 full pages + a tail of 8; request 1: 32 = 2 full pages
    return SimpleNamespace(spec=spec, seq_lens=np.array([40, 32], np.int32))


# lists per (request, KV head); request 0's lengths count its tail page
LENGTHS = np.array([[[2, 3], [1, 2]]], np.int32)


def test_step_bytes_by_hand():
    w = _workload()
    layer, total, pages_read, parts = bench.step_bytes(w, LENGTHS, 0.99)
    # tokens: request 0 keeps 1 and 2 full pages plus the 8-token tail, request 1
    # keeps 1 and 2 full pages: 24 + 40 + 16 + 32 = 112 tokens of K and V
    kv = 112 * 128 * 2 * 2
    summaries = 4 * (2 * 128 * 2)              # 4 full pages x 2 KV heads x 256 B
    q = 2 * 8 * 128 * 2
    out = 2 * 8 * 128 * 4
    assert parts == {"summaries": summaries, "kv": kv, "q": q, "out": out}
    assert total == kv + summaries + q + out == int(layer.sum())
    assert pages_read == pytest.approx(8 / 10)  # 8 listed of (3 + 2) pages x 2 KV heads


def test_step_bytes_dense_reads_no_summaries():
    w = _workload()
    _, total, _, parts = bench.step_bytes(w, LENGTHS, 1.0)
    assert parts["summaries"] == 0
    assert total == parts["kv"] + parts["q"] + parts["out"]


def test_step_bytes_low_bit_records():
    w = _workload()
    _, _, _, parts = bench.step_bytes(w, LENGTHS, 0.99, summ_page_bytes=288)
    assert parts["summaries"] == 4 * 288        # one record per full page


def test_traffic_shape_threshold_matches_the_kernel():
    """The benchmark picks the DRAM-traffic figure of the attention kernel's
    block shape by the number of lists; its switch-over must be the kernel's."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(bench.__file__), "sparse_long_context_page_gb300", "csrc",
                            "attend_core.cuh")).read()
    m = re.search(r"constexpr int kManyUnits = (\d+);", src)
    assert m, "kManyUnits not found in attend_core.cuh"
    assert int(m.group(1)) == bench.ATTEND_TRAFFIC["many_lists_from"]
    assert set(bench.ATTEND_TRAFFIC["dram_bytes_per_entry"]) == {"few_lists", "many_lists"}
