"""moira_append_kv: one token per request written into the paged pools, and
the summary of every page that fills, against the oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

from oracle import oracle
import sparse_long_context_page_gb300 as moira

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

D, S = 128, 16


def u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _pools(P, Hkv, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    k = torch.randn((P, Hkv, S, D), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((P, Hkv, S, D), generator=g, device="cuda").to(torch.bfloat16)
    return k, v


def _summaries_of(k_host):
    P, Hkv = k_host.shape[:2]
    return oracle.summaries(k_host.reshape(-1, S, D)).reshape(P, Hkv, D)


def test_append_writes_tokens_and_summarises_filled_pages():
    P, Hkv, B, max_pages = 64, 2, 6, 8
    shape = moira.Shape.of(4 * Hkv, Hkv, P)
    k_pool, v_pool = _pools(P, Hkv, 1)
    summ = torch.zeros((P, Hkv, D), dtype=torch.bfloat16, device="cuda")
    moira.update_summaries(shape, k_pool, summ, torch.arange(P, dtype=torch.int32, device="cuda"))
    rng = np.random.default_rng(2)
    table = rng.permutation(P)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    # tokens after the append: fills page 2, starts page 2, middle of page 5,
    # nothing, fills page 0, the last slot of the last page
    lens = np.array([16 * 3, 16 * 2 + 1, 16 * 5 + 8, 0, 16, 16 * max_pages], np.int32)
    g = torch.Generator(device="cuda").manual_seed(3)
    k_new = torch.randn((B, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
    v_new = torch.randn((B, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
    k0, v0, s0 = u16(k_pool), u16(v_pool), u16(summ)
    moira.append_kv(shape, k_new, v_new, k_pool, v_pool, summ, torch.from_numpy(table).cuda(),
                    torch.from_numpy(lens).cuda())
    torch.cuda.synchronize()
    k_want, v_want, s_want = k0.copy(), v0.copy(), s0.copy()
    kn, vn = u16(k_new), u16(v_new)
    filled = []
    for r in range(B):
        if lens[r] == 0:
            continue
        pos = lens[r] - 1
        p = table[r, pos // S]
        k_want[p, :, pos % S] = kn[r]
        v_want[p, :, pos % S] = vn[r]
        if pos % S == S - 1:
            filled.append(p)
    for p in filled:
        s_want[p] = _summaries_of(k_want[p:p + 1])[0]
    assert np.array_equal(u16(k_pool), k_want)
    assert np.array_equal(u16(v_pool), v_want)
    assert np.array_equal(u16(summ), s_want)                      # bit-exact, untouched elsewhere
    assert len(filled) == 3


def test_append_decode_loop_matches_a_fresh_build():
    """Forty appends from a ragged start: the pools hold every token where a
    fresh build would put it, and every full page's summary equals the
    oracle's summary of the final pool."""
    P, Hkv, B, max_pages = 96, 4, 3, 24
    shape = moira.Shape.of(4 * Hkv, Hkv, P)
    k_pool, v_pool = _pools(P, Hkv, 5)
    rng = np.random.default_rng(6)
    table = rng.permutation(P)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    lens = np.array([16 * 2 + 5, 16 * 7, 1], np.int32)            # tokens already in the cache
    summ = torch.zeros((P, Hkv, D), dtype=torch.bfloat16, device="cuda")
    full0 = np.concatenate([table[r, :lens[r] // S] for r in range(B)]).astype(np.int32)
    moira.update_summaries(shape, k_pool, summ, torch.from_numpy(full0).cuda())
    pt = torch.from_numpy(table).cuda()
    g = torch.Generator(device="cuda").manual_seed(7)
    for step in range(40):
        lens = lens + 1
        k_new = torch.randn((B, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
        v_new = torch.randn((B, Hkv, D), generator=g, device="cuda").to(torch.bfloat16)
        moira.append_kv(shape, k_new, v_new, k_pool, v_pool, summ, pt, torch.from_numpy(lens).cuda())
        # the token landed where it belongs
        kh = u16(k_pool)
        for r in range(B):
            pos = lens[r] - 1
            assert np.array_equal(kh[table[r, pos // S], :, pos % S], u16(k_new)[r])
    torch.cuda.synchronize()
    kh, sh = u16(k_pool), u16(summ)
    for r in range(B):
        for lp in range(lens[r] // S):
            p = table[r, lp]
            assert np.array_equal(sh[p], _summaries_of(kh[p:p + 1])[0]), (r, lp)
