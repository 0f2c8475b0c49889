"""The page-summary kernel's exact sums, through the C ABI, against the oracle.

The kernel forms each dimension's sum of a page's 16 bf16 keys in fp32 when
the keys are normal, below 2^124 and their exponents span at most 12 (every
partial sum then fits 24 bits), with 64-bit integer adds of the keys'
significands when the exponents span at most 40 (every partial sum fits 53
bits), and with fp64 adds in token order otherwise; in each case the
oracle's fp64 sum in token order is exact and equal.  This pool is built so
that every path, and each edge between them, is taken: spreads of 0 to 120
bits across dimensions, zeros of both signs, subnormals, means that round to
subnormals from normal keys, exact cancellation, infinities, NaN, keys just
below and at the fp32 limit of 16 summed keys, and the largest finite keys.
Every summary in every format must match the oracle's bit for bit.
"""
import numpy as np
import pytest
import torch

import helpers as H
from oracle import oracle
from sparse_long_context_page_gb300 import _binding as mb

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():          # collected on CPU machines, never run there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

S, D, HKV = 16, 128, 8


def _bits(x):
    """fp32 values -> bf16 bit patterns (exact: every value here is a bf16)."""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _pool():
    rng = np.random.default_rng(42)
    pages = []
    normal = rng.standard_normal((HKV, S, D)).astype(np.float32)
    pages.append(_bits(normal))                                          # the usual keys
    pages.append(np.zeros((HKV, S, D), np.uint16))                       # +0
    pages.append(np.full((HKV, S, D), 0x8000, np.uint16))                # -0
    x = _bits(rng.standard_normal((HKV, S // 2, D)).astype(np.float32))
    pages.append(np.concatenate([x, x ^ np.uint16(0x8000)], axis=1))     # x and -x cancel
    # dimension d: keys 2^a and 2^(a - spread), spread = d (0 .. 127 bits),
    # straddling the 40-bit edge of the integer path
    sp = np.zeros((HKV, S, D), np.float32)
    for d in range(D):
        spread = d if d < 64 else d - 64 + 30
        a = 60 - (spread // 2)
        sp[:, 0, d] = 2.0 ** a
        sp[:, 1, d] = -(2.0 ** (a - spread))
        sp[:, 2:, d] = rng.standard_normal((HKV, S - 2)).astype(np.float32) * 2.0 ** (a - spread // 3)
    pages.append(_bits(sp))
    sub = np.zeros((HKV, S, D), np.uint16)
    sub[:, :, : D // 2] = rng.integers(1, 128, (HKV, S, D // 2))         # subnormals only
    sub[:, :, D // 2:] = rng.integers(1, 128, (HKV, S, D // 2))
    sub[:, 0, D // 2:] = _bits(np.full((HKV, D // 2), 3.0))             # with a normal key: wide spread
    pages.append(sub)
    special = _bits(rng.standard_normal((HKV, S, D)).astype(np.float32))
    special[0, 3, 5] = 0x7F80                                            # +inf
    special[1, 7, 9] = 0x7FC0                                            # NaN
    special[2, 1, 11], special[2, 2, 11] = 0x7F80, 0xFF80                # +inf and -inf
    pages.append(special)
    big = np.full((HKV, S, D), 0x7F7F, np.uint16)                        # the largest finite bf16
    big[:, ::2, :] ^= np.uint16(0x8000)
    big[:, 0, : D // 2] = 0x7F7F
    pages.append(big)
    ext = np.zeros((HKV, S, D), np.uint16)
    ext[:, 0, :] = 0x7F00                                                # 2^127
    ext[:, 1, :] = 0x0001                                                # 2^-133
    ext[:, 2:, :] = _bits(rng.standard_normal((HKV, S - 2, D)).astype(np.float32))
    pages.append(ext)
    # 16 keys of one sign at exponent field 250 (the fp32 sum stays finite) and
    # 251 (it would not), per head and dimension a random significand
    for e in (250, 251):
        lim = np.uint16(e << 7) | rng.integers(0, 128, (HKV, S, D)).astype(np.uint16)
        lim[:, :, D // 2:] |= np.uint16(0x8000)
        pages.append(lim)
    # the smallest normal exponents: means below 2^-126 round to bf16 subnormals
    tiny = (rng.integers(1, 8, (HKV, S, D)) << 7 | rng.integers(0, 128, (HKV, S, D))).astype(np.uint16)
    tiny[:, 1::2, :] ^= np.uint16(0x8000)
    pages.append(tiny)
    return np.stack(pages)                                               # [P][Hkv][S][d]


@pytest.mark.parametrize("fmt", [mb.SUMM_BF16, mb.SUMM_Q8, mb.SUMM_Q2])
def test_summaries_take_both_sum_paths_bit_exact(fmt):
    k = _pool()
    P = k.shape[0]
    k_dev = torch.from_numpy(k.view(np.int16)).cuda().view(torch.bfloat16)
    shape = mb.Shape.of(4 * HKV, HKV, P)
    summ = mb.make_summaries(shape, fmt, device="cuda")
    pages = torch.arange(P, dtype=torch.int32, device="cuda")
    for _ in range(2):                                                   # twice: nothing left over
        mb.update_summaries(shape, k_dev, summ, pages, fmt=fmt)
        torch.cuda.synchronize()
        if fmt == mb.SUMM_BF16:
            got = H.u16(summ)
            ref = oracle.summaries(k.reshape(-1, S, D)).reshape(P, HKV, D)
            diff = np.argwhere(got != ref)
            assert len(diff) == 0, f"{len(diff)} summary elements differ, first (page, head, dim) {diff[:4]}"
        else:
            bits = 8 if fmt == mb.SUMM_Q8 else 2
            codes, steps = oracle.summaries_lowbit(k.reshape(-1, S, D), bits)
            ref = H.pack_lowbit(codes.reshape(P, HKV, D), steps.reshape(P, HKV), bits,
                                mb.summary_page_bytes(shape, fmt))
            got = summ.cpu().numpy()
            assert np.array_equal(got, ref), f"{int((got != ref).sum())} record bytes differ"
