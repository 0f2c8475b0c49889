// Selection arithmetic shared by k_select (one block per list) and
// k_select_attend (the lists of a small batch selected by many blocks each,
// then attended in the same launch).  Both must reach the same lists bit for
// bit, so the page masses and the cut come from these functions only.
//
// The estimate ("MOIRA: Mass-Oriented Indexing with Ragged Attention for
// Long-Context Decoding", abstract: pages are chosen by their estimated
// attention mass), with k_score's per-chunk statistics (M_c, Z_c) and
// chunk-relative weights e_hp = 2^(s_hp - M_c) in the log2 domain:
//   M_h = max_c M_c,  Z_h = sum_c 2^(M_c - M_h) Z_c,
//   m_p = sum_h e_hp * 2^(M_c - M_h) / (G Z_h)  = (1/G) sum_h softmax_p(s_h.)
// Coverage keeps the fewest pages, heaviest first (lower logical index first
// among equal masses), whose masses reach gamma.  The masses enter the cut as
// 2^-31 fixed-point integers, so every sum is exact and the cut does not
// depend on the order in which blocks or threads add them.
#pragma once

#include "moira_device.cuh"
#include "moira_launch.h"

namespace moira {

// Level-1 bins: the fp32 bit pattern >> 16 (exponent + 7 fraction bits, 128
// bins per octave) for masses in [2^-32, 2); bin 0 gathers everything below
// (kKeyLo, kL1Bins: moira_device.cuh).
__device__ __forceinline__ int l1_bin(uint32_t x)
{
    const uint32_t k = x >> 16;
    return k < kKeyLo ? 0 : static_cast<int>(k - kKeyLo) + 1;
}
__device__ __forceinline__ uint32_t l1_lo(int b) { return b == 0 ? 0u : (static_cast<uint32_t>(b - 1) + kKeyLo) << 16; }
__device__ __forceinline__ uint32_t l1_hi(int b) { return b == 0 ? (kKeyLo << 16) : (static_cast<uint32_t>(b) + kKeyLo) << 16; }

// Mass as a 2^-31 fixed-point integer.  Masses sum to 1 (to fp32 rounding),
// so every histogram bin and every partial sum fits in 32 bits; rounding each
// mass costs at most 2^-32, i.e. < 1e-5 over 16384 pages.
__device__ __forceinline__ uint32_t to_fx(uint32_t x)
{
    return __float2uint_rn(__uint_as_float(x) * 0x1p31f);
}

// What a page adds to the histograms: its fixed-point mass for the coverage
// rule, 1 for top-k (the descent then counts pages instead of mass).
__device__ __forceinline__ uint32_t rule_weight(int rule, uint32_t x)
{
    return rule == kRuleTopK ? 1u : to_fx(x);
}

constexpr int kPairMax = 256;               // crossing-bin pages resolved pairwise

// One refinement level of the cut inside [lo, hi): the bins of width 2^shift
// (nb of them, at most kL2Bins) are read through bin(i) by one warp, lane l
// owning bins nb-1-8l .. nb-8-8l from the top; starting from `above` (the
// fixed-point mass of everything at or above hi), the bin in which the running
// sum reaches `target` becomes the new [lo, hi) and `above` the mass above
// it.  Returns false if no bin reaches the target (cannot happen with exact
// sums of a range that was chosen because it reaches it).  Every lane of the
// warp calls it and gets the same result.
template <class Bin>
__device__ __forceinline__ bool warp_pick_bin(Bin bin, int nb, int shift, unsigned long long target,
                                              uint32_t &lo, uint32_t &hi, unsigned long long &above)
{
    const int lane = threadIdx.x & 31;
    const int top = nb - 1 - 8 * lane;
    uint32_t hv[8];
    unsigned long long mine = 0ull;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        hv[i] = top - i >= 0 ? bin(top - i) : 0u;
        mine += hv[i];
    }
    unsigned long long xs = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, xs, o);
        if (lane >= o) xs += y;
    }
    unsigned long long acc = above + xs - mine;
    int fb = -1;
    unsigned long long fa = 0ull;
    if (acc < target && acc + mine >= target) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int b = top - i;
            if (b < 0) break;
            if (acc + hv[i] >= target) {
                fb = b;
                fa = acc;
                break;
            }
            acc += hv[i];
        }
    }
    const unsigned who = __ballot_sync(0xffffffffu, fb >= 0);
    if (!who) return false;
    const int src = __ffs(who) - 1;
    fb = __shfl_sync(0xffffffffu, fb, src);
    above = __shfl_sync(0xffffffffu, fa, src);
    const uint32_t nlo = lo + (static_cast<uint32_t>(fb) << shift);
    const uint32_t span = 1u << shift;
    hi = (hi - nlo < span) ? hi : nlo + span;
    lo = nlo;
    return true;
}

// Bin width of the next refinement level of [lo, hi): at most kL2Bins bins.
__device__ __forceinline__ void refine_bins(uint32_t lo, uint32_t hi, int &shift, int &nb)
{
    const uint32_t width = hi - lo;
    const int nbits = 32 - __clz(width - 1u);
    shift = nbits > 8 ? nbits - 8 : 0;
    nb = static_cast<int>((width - 1u) >> shift) + 1;
}

// The cut inside the crossing bin [lo, hi) from its pages' mass bit patterns
// cand[0 .. nc) (shared memory), by one warp: 256-bin radix levels over the
// candidates until one bit pattern is left.  h2: kL2Bins words of shared
// scratch.  Every lane calls it; lo, hi and above are updated in place.
__device__ __forceinline__ void warp_refine(const uint32_t *cand, int nc, uint32_t *h2, int rule,
                                            unsigned long long target, uint32_t &lo, uint32_t &hi,
                                            unsigned long long &above)
{
    const int lane = threadIdx.x & 31;
    for (int pass = 0; hi - lo > 1u && pass < 6; ++pass) {
        int shift, nb;
        refine_bins(lo, hi, shift, nb);
#pragma unroll
        for (int i = 0; i < kL2Bins / 32; ++i) h2[lane + 32 * i] = 0u;
        __syncwarp();
        for (int c = lane; c < nc; c += 32) {
            const uint32_t x = cand[c];
            if (x >= lo && x < hi) atomicAdd(&h2[(x - lo) >> shift], rule_weight(rule, x));
        }
        __syncwarp();
        const bool ok = warp_pick_bin([&](int b) { return h2[b]; }, nb, shift, target, lo, hi, above);
        __syncwarp();
        if (!ok) break;                           // cannot happen: exact integer sums
    }
}

// The normaliser reduction, in a fixed order: per head, 8 lanes-of-32 groups
// ("virtual warps") each hold the chunks w*32 + lane and w*32 + lane + 256;
// a virtual warp's sum is its butterfly (xor 16, 8, 4, 2, 1) and the head's
// Z is the 8 group sums added in order.  The maximum needs no fixed order.
__device__ __forceinline__ float chunk_weight_sum(float cm0, float cz0, float cm1, float cz1, float M)
{
    const float e0 = cm0 == -INFINITY ? 0.f : exp2f(cm0 - M);
    const float e1 = cm1 == -INFINITY ? 0.f : exp2f(cm1 - M);
    return fmaf(cz1, e1, fmaf(cz0, e0, 0.f));
}

__device__ __forceinline__ float warp_sum_butterfly(float z)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    return z;
}

__device__ __forceinline__ float warp_max_butterfly(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// 1 / (G Z) of a head from its 8 group sums, added in order.
__device__ __forceinline__ float head_zinv(const float *group_sums)
{
    float Z = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) Z += group_sums[w];
    return Z > 0.f ? 1.f / (kGroup * Z) : 0.f;
}

// A chunk's factor 2^(M_c - M_h) / (G Z_h).
__device__ __forceinline__ float chunk_factor(float cm, float M, float zinv)
{
    return (cm == -INFINITY ? 0.f : exp2f(cm - M)) * zinv;
}

// A page's mass from its 4 heads' chunk-relative weights and the chunk
// factors f = (f_h0, f_h1, f_h2, f_h3), as the fp32 bit pattern of the mass
// clamped to [0, 1.5] (NaN -> 0): for non-negative floats the patterns order
// like the values.
__device__ __forceinline__ uint32_t page_mass_bits(float w0, float w1, float w2, float w3, float4 f)
{
    const float m = fmaf(w3, f.w, fmaf(w2, f.z, fmaf(w1, f.y, w0 * f.x)));
    return __float_as_uint(fminf(fmaxf(m, 0.f), 1.5f));
}

}  // namespace moira
