"""Seeded synthetic decode workloads for the sparse-decode path.

This module only draws inputs: queries, paged K/V caches, page tables and
sequence lengths.  It holds none of the method's arithmetic (no summaries,
scores, masses, selection or attention), so the CUDA library and the CPU
oracle can both be fed from it.

The pages measure on RULER at 128k context with a real model; neither the
suite nor trained weights exist here, so these inputs stand in for them with
the shapes of a Llama-3-8B-style model (32 layers, 32 query / 8 KV heads,
head dim 128, 16-token pages) and keys whose attention mass is concentrated
on a few planted pages by a controllable amount.

Recipe (all draws seeded):
  * small draws (queries, concentrations, planted pages, sequence lengths,
    page-table permutation, regimes) come from ``numpy.random.default_rng``,
    so they are identical on every device;
  * the bulk N(0, 1) key/value noise comes from a ``torch.Generator`` on the
    target device (values therefore differ between CPU and CUDA runs, the
    structure does not);
  * q_h = sqrt(d) * unit(N(0, I_d)) per query head, stored bf16;
  * qhat_j = sqrt(d) * unit(sum of the group's bf16 queries) for KV head j;
  * a "planted" page with concentration c has every key = c * qhat_j + N(0, I);
  * V ~ N(0, 1) everywhere; every tensor on the device is bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class WorkloadSpec:
    name: str
    batch: int
    layers: int
    q_heads: int
    kv_heads: int
    context: tuple            # per-request token counts; () with loguniform=True
    gammas: tuple
    keys: str                 # "planted_fixed" | "planted_random" | "regimes"
    head_dim: int = 128
    page_size: int = 16
    loguniform: tuple = ()    # (lo, hi) token range for ragged batches
    n_planted: int = 8        # planted_fixed only
    c_fixed: float = 3.0      # planted_fixed only


SPECS = {
    # 1 request, 1 layer, 8/2 heads, 4096 tokens; 8 planted pages per KV head, c = 3.
    "tiny": WorkloadSpec("tiny", 1, 1, 8, 2, (4096,), (0.9, 0.99, 1.0), "planted_fixed"),
    # Llama-3-8B-shaped single request at 32k; per (layer, KV head) c ~ U[0,4] on 1-5% of pages.
    "llama8b_32k": WorkloadSpec("llama8b_32k", 1, 32, 32, 8, (32768,), (0.99,), "planted_random"),
    # The same at 128k context (8192 pages per KV head): the headline decode step.
    "llama8b_128k": WorkloadSpec("llama8b_128k", 1, 32, 32, 8, (131072,), (0.98, 0.99, 1.0),
                                 "planted_random"),
    # 32 concurrent requests, lengths log-uniform in [8192, 131072], randomly permuted pool.
    "serving_ragged": WorkloadSpec("serving_ragged", 32, 32, 32, 8, (), (0.99,), "planted_random",
                                   loguniform=(8192, 131072)),
    # 64 requests at 64k, one layer; per KV head a flat, dominant-page or heavy-tail regime.
    "stress_regimes": WorkloadSpec("stress_regimes", 64, 1, 32, 8, (65536,) * 64, (0.99,), "regimes"),
}

REGIMES = ("flat", "dominant", "heavy")


@dataclass
class Workload:
    spec: WorkloadSpec
    seed: int
    seq_lens: np.ndarray          # int32 [B]
    page_table: np.ndarray        # int32 [B][max_pages], -1 past each request's pages
    num_phys_pages: int           # P, pages in the pool of every layer
    q: torch.Tensor               # bf16 [Lyr][B][Hq][d]
    k_pool: torch.Tensor          # bf16 [Lyr][P][Hkv][S][d]
    v_pool: torch.Tensor          # bf16 [Lyr][P][Hkv][S][d]
    info: dict = field(default_factory=dict)   # per-unit generation facts (c, planted, regime)

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def group(self) -> int:
        return self.spec.q_heads // self.spec.kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.head_dim)

    def pages_of(self, r: int) -> int:
        L = int(self.seq_lens[r])
        S = self.spec.page_size
        return L // S + (L % S != 0)


def spec(name: str, **overrides) -> WorkloadSpec:
    """A named spec, optionally with fields replaced (e.g. fewer layers)."""
    return replace(SPECS[name], **overrides) if overrides else SPECS[name]


def _seq_lens(sp: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    if sp.loguniform:
        lo, hi = sp.loguniform
        u = rng.uniform(math.log(lo), math.log(hi), size=sp.batch)
        return np.floor(np.exp(u)).astype(np.int32)
    ctx = list(sp.context)
    if len(ctx) == 1:
        ctx = ctx * sp.batch
    assert len(ctx) == sp.batch
    return np.asarray(ctx, np.int32)


def _queries(sp: WorkloadSpec, rng: np.random.Generator) -> np.ndarray:
    d = sp.head_dim
    q = rng.standard_normal((sp.layers, sp.batch, sp.q_heads, d))
    q = q / np.linalg.norm(q, axis=-1, keepdims=True) * math.sqrt(d)
    return q.astype(np.float32)


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)


# Rows of fp32 noise generated per call; fixed so that the stream of draws
# does not depend on the size of the workload's other dimensions.
_NOISE_CHUNK_PAGES = 4096


def _noise_bf16(shape, gen, device, add=None):
    """N(0,1) draws of ``shape`` (pages first), optionally plus fp32 offsets,
    rounded once to bf16.  ``add(lo, hi, chunk)`` may modify the fp32 chunk."""
    P = shape[0]
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    for lo in range(0, P, _NOISE_CHUNK_PAGES):
        hi = min(P, lo + _NOISE_CHUNK_PAGES)
        ch = torch.randn((hi - lo,) + tuple(shape[1:]), generator=gen, device=device,
                         dtype=torch.float32)
        if add is not None:
            add(lo, hi, ch)
        out[lo:hi] = ch.to(torch.bfloat16)
    return out


def make_workload(name_or_spec, seed: int = 0, device="cuda", max_pages: int | None = None,
                  **overrides) -> Workload:
    """Draw one workload.  ``overrides`` replace spec fields (sizes for tests)."""
    sp = name_or_spec if isinstance(name_or_spec, WorkloadSpec) else spec(name_or_spec, **overrides)
    if isinstance(name_or_spec, WorkloadSpec) and overrides:
        sp = replace(sp, **overrides)
    device = torch.device(device)
    rng = np.random.default_rng(seed)
    B, Lyr, Hq, Hkv, d, S = sp.batch, sp.layers, sp.q_heads, sp.kv_heads, sp.head_dim, sp.page_size
    G = Hq // Hkv

    seq_lens = _seq_lens(sp, rng)
    n_pages = [int(L) // S + (int(L) % S != 0) for L in seq_lens]
    P = max(1, sum(n_pages))
    mp = max(n_pages) if max_pages is None else max_pages
    assert mp >= max(n_pages)
    perm = rng.permutation(P).astype(np.int32)
    page_table = np.full((B, max(mp, 1)), -1, np.int32)
    off = 0
    for r in range(B):
        page_table[r, :n_pages[r]] = perm[off:off + n_pages[r]]
        off += n_pages[r]

    qf = _queries(sp, rng)
    q = _bf16(qf)                                           # [Lyr][B][Hq][d]
    qr = q.float().numpy().reshape(Lyr, B, Hkv, G, d)       # the stored queries
    qsum = qr.sum(axis=3)
    qhat = qsum / np.linalg.norm(qsum, axis=-1, keepdims=True) * math.sqrt(d)   # [Lyr][B][Hkv][d]

    # Per-unit key structure: a list of (logical page, fp32 offset vector, replace?) per unit.
    info = {"c": np.zeros((Lyr, B, Hkv)), "planted": np.zeros((Lyr, B, Hkv), np.int64),
            "regime": np.full((Lyr, B, Hkv), "", dtype=object)}
    plants = []      # (layer, r, j, logical pages array, offset rows [n][d] fp32, replace)
    for l in range(Lyr):
        for r in range(B):
            F = int(seq_lens[r]) // S
            for j in range(Hkv):
                if F == 0:
                    continue
                if sp.keys == "planted_fixed":
                    c = sp.c_fixed
                    pages = rng.choice(F, size=min(sp.n_planted, F), replace=False)
                    plants.append((l, r, j, pages, np.repeat(c * qhat[l, r, j][None], len(pages), 0), False))
                    info["c"][l, r, j], info["planted"][l, r, j] = c, len(pages)
                elif sp.keys == "planted_random":
                    c = rng.uniform(0.0, 4.0)
                    frac = rng.uniform(0.01, 0.05)
                    k = max(1, int(round(frac * F)))
                    pages = rng.choice(F, size=k, replace=False)
                    plants.append((l, r, j, pages, np.repeat(c * qhat[l, r, j][None], k, 0), False))
                    info["c"][l, r, j], info["planted"][l, r, j] = c, k
                elif sp.keys == "regimes":
                    reg = REGIMES[int(rng.integers(3))]
                    info["regime"][l, r, j] = reg
                    if reg == "dominant":
                        p = np.array([int(rng.integers(F))])
                        plants.append((l, r, j, p, 8.0 * qhat[l, r, j][None], True))
                        info["planted"][l, r, j] = 1
                    elif reg == "heavy":
                        rho = rng.permutation(F) + 1            # ranks 1..F
                        beta = -1.1 * np.log(rho)               # Zipf(1.1) log-weights
                        kappa = float(np.mean(qr[l, r, j] @ qhat[l, r, j])) / math.sqrt(d)
                        offs = beta[:, None] * qhat[l, r, j][None] / kappa
                        plants.append((l, r, j, np.arange(F), offs, False))
                        info["planted"][l, r, j] = F
                else:
                    raise ValueError(sp.keys)

    gen = torch.Generator(device=device)
    k_pool = torch.empty((Lyr, P, Hkv, S, d), dtype=torch.bfloat16, device=device)
    v_pool = torch.empty((Lyr, P, Hkv, S, d), dtype=torch.bfloat16, device=device)
    for l in range(Lyr):
        # one flat list of (physical page, head, offset, replace) for this layer
        rows_phys, rows_head, rows_off, rows_rep = [], [], [], []
        for (ll, r, j, pages, offs, rep) in plants:
            if ll != l:
                continue
            rows_phys.append(page_table[r, pages])
            rows_head.append(np.full(len(pages), j, np.int64))
            rows_off.append(offs.astype(np.float32))
            rows_rep.append(np.full(len(pages), rep, bool))
        if rows_phys:
            phys = np.concatenate(rows_phys).astype(np.int64)
            head = np.concatenate(rows_head)
            offv = np.concatenate(rows_off)
            repv = np.concatenate(rows_rep)
            order = np.argsort(phys, kind="stable")
            phys, head, offv, repv = phys[order], head[order], offv[order], repv[order]
        else:
            phys = np.zeros(0, np.int64)
        t_phys = torch.from_numpy(phys).to(device) if len(phys) else None

        def add(lo, hi, ch, phys=phys, head=head if len(phys) else None,
                offv=offv if len(phys) else None, repv=repv if len(phys) else None):
            if not len(phys):
                return
            a, b = np.searchsorted(phys, lo), np.searchsorted(phys, hi)
            if a == b:
                return
            pi = torch.from_numpy(phys[a:b] - lo).to(device)
            hi_ = torch.from_numpy(head[a:b]).to(device)
            ov = torch.from_numpy(offv[a:b]).to(device)[:, None, :]     # [n][1][d]
            rp = torch.from_numpy(repv[a:b]).to(device)[:, None, None]
            cur = ch[pi, hi_]                                           # [n][S][d]
            ch[pi, hi_] = torch.where(rp, ov.expand_as(cur), cur + ov)

        gen.manual_seed(int(seed) * 1_000_003 + 2 * l)
        k_pool[l] = _noise_bf16((P, Hkv, S, d), gen, device, add)
        gen.manual_seed(int(seed) * 1_000_003 + 2 * l + 1)
        v_pool[l] = _noise_bf16((P, Hkv, S, d), gen, device)
        del t_phys

    return Workload(spec=sp, seed=seed, seq_lens=seq_lens, page_table=page_table,
                    num_phys_pages=P, q=q.to(device), k_pool=k_pool, v_pool=v_pool, info=info)


def random_lists(w: Workload, seed: int, keep_frac=(0.0, 1.0)):
    """Seeded page lists that follow the selection contract, for testing
    attention on its own: per (request, KV head) a random subset of the full
    pages (ascending logical order) plus the partial tail page last.
    Returns (logical lists as a list of arrays [B][Hkv], physical int32
    [B][Hkv][max_pages], lengths int32 [B][Hkv])."""
    rng = np.random.default_rng(seed)
    B, Hkv, S = w.spec.batch, w.spec.kv_heads, w.spec.page_size
    logical = []
    phys = np.full((B, Hkv, w.max_pages), -1, np.int32)
    lengths = np.zeros((B, Hkv), np.int32)
    for r in range(B):
        L = int(w.seq_lens[r])
        F, T = L // S, int(L % S != 0)
        row = []
        for j in range(Hkv):
            f = rng.uniform(*keep_frac)
            keep = np.flatnonzero(rng.random(F) < f)
            lst = np.concatenate([keep, [F]] if T else [keep]).astype(np.int32)
            row.append(lst)
            phys[r, j, :len(lst)] = w.page_table[r, lst]
            lengths[r, j] = len(lst)
        logical.append(row)
    return logical, phys, lengths
