"""Device buffers for one decode workload, driven through the C ABI.

Holds the per-layer summaries, page table, lists, lengths, outputs and the
workspace that ``moira_select`` / ``moira_attend`` need, so that a caller can
run a whole decode-attention step with one call (or capture it in a graph).
"""
from __future__ import annotations

import torch

from . import _binding as mb
from .workloads import Workload


class DecodeState:
    """`fmt` picks the page-summary format (mb.SUMM_BF16 / SUMM_Q8 / SUMM_Q2)."""

    def __init__(self, w: Workload, max_pages: int | None = None, fmt: int = mb.SUMM_BF16):
        sp = w.spec
        dev = w.q.device
        self.w = w
        self.device = dev
        self.layers, self.batch = sp.layers, sp.batch
        self.max_pages = w.max_pages if max_pages is None else max_pages
        self.shape = mb.Shape.of(sp.q_heads, sp.kv_heads, w.num_phys_pages)
        self.sm_scale = w.sm_scale
        pt = torch.full((sp.batch, self.max_pages), -1, dtype=torch.int32)
        pt[:, :w.max_pages] = torch.from_numpy(w.page_table)
        self.page_table = pt.to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.fmt = fmt
        self.summ = mb.make_summaries(self.shape, fmt, layers=sp.layers, device=dev)
        self.lists = torch.zeros((sp.batch, sp.kv_heads, self.max_pages), dtype=torch.int32, device=dev)
        self.lengths = torch.zeros((sp.layers, sp.batch, sp.kv_heads), dtype=torch.int32, device=dev)
        self.out = torch.zeros((sp.layers, sp.batch, sp.q_heads, sp.head_dim), dtype=torch.float32,
                               device=dev)
        self.ws = mb.make_workspace(self.shape, sp.batch, self.max_pages, device=dev)

    def summarize(self):
        """Summaries of every physical page of every layer (after prefill)."""
        pages = torch.arange(self.w.num_phys_pages, dtype=torch.int32, device=self.device)
        for l in range(self.layers):
            mb.update_summaries(self.shape, self.w.k_pool[l], self.summ[l], pages, fmt=self.fmt)

    def step(self, gamma: float):
        """One decode-attention step over all layers (select + attend per layer)."""
        if self.fmt == mb.SUMM_BF16:
            mb.decode_step(self.shape, self.w.q, self.w.k_pool, self.w.v_pool, self.summ,
                           self.page_table, self.seq_lens, gamma, self.sm_scale, self.lists,
                           self.lengths, self.out, self.ws)
        else:
            mb.decode_step_ex(self.shape, self.fmt, self.w.q, self.w.k_pool, self.w.v_pool,
                              self.summ, self.page_table, self.seq_lens, mb.RULE_COVERAGE, gamma,
                              self.sm_scale, self.lists, self.lengths, self.out, self.ws)

    def step_rule(self, rule: int, param: float):
        """One decode-attention step under a page rule: per layer moira_select_rule
        then moira_attend, in order on the current stream."""
        for l in range(self.layers):
            self.select_layer_rule(l, rule, param, self.lists, self.lengths[l])
            self.attend_layer(l, self.lists, self.lengths[l], self.out[l])

    def select_layer(self, l: int, gamma: float, lists=None, lengths=None):
        lists = self.lists if lists is None else lists
        lengths = self.lengths[l] if lengths is None else lengths
        if self.fmt == mb.SUMM_BF16:
            mb.select(self.shape, self.w.q[l], self.summ[l], self.page_table, self.seq_lens, gamma,
                      self.sm_scale, lists, lengths, self.ws)
        else:
            mb.select_ex(self.shape, self.fmt, self.w.q[l], self.summ[l], self.page_table,
                         self.seq_lens, mb.RULE_COVERAGE, gamma, self.sm_scale, lists, lengths, self.ws)
        return lists, lengths

    def select_layer_clustered(self, l: int, gamma: float, lists=None, lengths=None):
        """moira_select_clustered on layer l (bf16 summaries only)."""
        lists = self.lists if lists is None else lists
        lengths = self.lengths[l] if lengths is None else lengths
        mb.select_clustered(self.shape, self.w.q[l], self.summ[l], self.page_table, self.seq_lens, gamma,
                            self.sm_scale, lists, lengths, self.ws)
        return lists, lengths

    def select_layer_rule(self, l: int, rule: int, param: float, lists=None, lengths=None):
        lists = self.lists if lists is None else lists
        lengths = self.lengths[l] if lengths is None else lengths
        if self.fmt == mb.SUMM_BF16:
            mb.select_rule(self.shape, self.w.q[l], self.summ[l], self.page_table, self.seq_lens,
                           rule, param, self.sm_scale, lists, lengths, self.ws)
        else:
            mb.select_ex(self.shape, self.fmt, self.w.q[l], self.summ[l], self.page_table,
                         self.seq_lens, rule, param, self.sm_scale, lists, lengths, self.ws)
        return lists, lengths

    def select_attend_layer(self, l: int, gamma: float, lists=None, lengths=None, out=None):
        """One layer's coverage selection and attention in one call
        (moira_select_attend, in this state's summary format)."""
        lists = self.lists if lists is None else lists
        lengths = self.lengths[l] if lengths is None else lengths
        out = self.out[l] if out is None else out
        mb.select_attend(self.shape, self.w.q[l], self.summ[l], self.w.k_pool[l], self.w.v_pool[l],
                         self.page_table, self.seq_lens, gamma, self.sm_scale, lists, lengths, out, self.ws,
                         fmt=self.fmt)
        return lists, lengths, out

    def score_layer(self, l: int):
        """The page-scoring kernel of layer l alone (results stay in the workspace)."""
        mb.score(self.shape, self.w.q[l], self.summ[l], self.page_table, self.seq_lens, self.sm_scale,
                 self.ws, fmt=self.fmt)

    def attend_layer(self, l: int, lists, lengths, out=None):
        out = self.out[l] if out is None else out
        mb.attend(self.shape, self.w.q[l], self.w.k_pool[l], self.w.v_pool[l], lists, lengths,
                  self.seq_lens, self.max_pages, self.sm_scale, out, self.ws)
        return out

    def device_status(self) -> int:
        return mb.read_device_status(self.ws)
