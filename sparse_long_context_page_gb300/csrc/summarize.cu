// Page summaries: the bf16 mean key of every (page, KV head) block.
//
// "MOIRA: Mass-Oriented Indexing with Ragged Attention for Long-Context
// Decoding", abstract: the coverage rule works on an *estimated* attention
// mass per page, which needs per-page metadata.  The form used here is the
// mean vector of the page's keys, one of the block summaries named in
// "Faster Flash Decoding", section 2 (related work).
//
// The mean of the 16 keys is their fp64 sum in token order divided by 16,
// rounded once to bf16, ties to even.  Wherever that sum is exact it is
// formed without fp64, whose rate on this GPU is far below what the HBM
// stream of keys needs: in fp32 when the keys' exponents span at most 12
// (every partial sum then fits 24 bits), else with 64-bit integer adds of
// the keys' significands when they span at most 40 (page_dim_sum_fixed),
// rounded to bf16 by integer arithmetic; only wider spreads, infinities and
// NaNs take fp64 adds in token order.  All three give the bits of the fp64
// sum.
//
// Low-bit formats store the same fp64 mean in 8 or 2 bits per element with
// the symmetric mid-rise quantiser that "Faster Flash Decoding", section 3.1,
// uses for its low-bit key thumbnails: one fp32 step per (page, KV head),
//   step = max_i |mean_i| / (2^(bits-1) - 1/2)   (fp64, rounded once to fp32)
//   code = floor(mean_i / step), clamped to [-2^(bits-1), 2^(bits-1) - 1]
// standing for (code + 1/2) * step; no zero level, so signs survive.  A
// non-finite mean element, a zero mean or a step that rounds to 0 gives
// step 0 and codes 0.
#include <cuda_bf16.h>

#include "moira_device.cuh"
#include "moira_launch.h"

namespace moira {

// Round a double to the nearest bf16 (ties to even) in one step, by integer
// arithmetic on the binary64 encoding: keep sign, exponent and the top 7
// fraction bits, adding half an ulp minus one plus the kept lsb before
// truncating.  Magnitudes below 2^-126 land on the bf16 subnormal grid
// (multiples of 2^-133), reached by exact scaling and rint().
__device__ __forceinline__ uint32_t f64_to_bf16_rne(double x)
{
    const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
    const uint32_t sign = static_cast<uint32_t>(u >> 48) & 0x8000u;
    const unsigned long long a = u & 0x7FFFFFFFFFFFFFFFull;
    if (a > 0x7FF0000000000000ull) return 0x7FC0u;                  // NaN
    const int biased = static_cast<int>(a >> 52);
    if (biased >= 1023 - 126) {                                       // |x| >= 2^-126
        const unsigned long long r = a + ((1ull << 44) - 1ull) + ((a >> 45) & 1ull);
        const int e_bf = static_cast<int>(r >> 52) - 1023 + 127;
        if (e_bf >= 255) return sign | 0x7F80u;                       // overflow / inf
        return sign | (static_cast<uint32_t>(e_bf) << 7) | static_cast<uint32_t>((r >> 45) & 0x7Full);
    }
    const double grid = rint(fabs(x) * 0x1p133);                      // in [0, 128]
    return sign | static_cast<uint32_t>(grid);
}

// Write the low-bit summary of KV head j of one page into its record `rec`
// from this thread's two fp64 means (dimensions 2*tid, 2*tid+1).  Called by
// all 64 threads of the block (it synchronises them); the block of the first
// head of each head group also zeroes that group's padding.
template <int kBits>
__device__ void store_lowbit(double lo, double hi, uint8_t *rec, int j, int hkv)
{
    __shared__ double s_a[2];
    __shared__ int s_bad[2];
    constexpr int kCb = lowbit_code_bytes(kBits);
    constexpr double kHalf = static_cast<double>(1 << (kBits - 1));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool bad = !isfinite(lo) || !isfinite(hi);
    double a = bad ? 0.0 : fmax(fabs(lo), fabs(hi));
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmax(a, __shfl_xor_sync(0xffffffffu, a, o));
    const bool any_bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
        s_a[warp] = a;
        s_bad[warp] = any_bad;
    }
    __syncthreads();
    a = fmax(s_a[0], s_a[1]);
    const float step = (s_bad[0] | s_bad[1]) ? 0.f : __double2float_rn(a / (kHalf - 0.5));
    int c0 = 0, c1 = 0;
    if (step > 0.f) {
        c0 = static_cast<int>(fmin(fmax(floor(lo / static_cast<double>(step)), -kHalf), kHalf - 1.0));
        c1 = static_cast<int>(fmin(fmax(floor(hi / static_cast<double>(step)), -kHalf), kHalf - 1.0));
    }
    const int gh = lowbit_group_heads(hkv), jj = j % gh;
    uint8_t *grp = rec + (j / gh) * lowbit_group_bytes(kBits, hkv);
    if constexpr (kBits == 8) {
        *reinterpret_cast<uint16_t *>(grp + jj * kCb + 2 * tid) =
            static_cast<uint16_t>((c0 & 0xFF) | ((c1 & 0xFF) << 8));
    } else {
        // element i sits in bits 2*(i%4) of byte i/4: this thread's pair is
        // one nibble, the low nibble for even tid
        const uint32_t nib = static_cast<uint32_t>(c0 + 2) | (static_cast<uint32_t>(c1 + 2) << 2);
        const uint32_t up = __shfl_down_sync(0xffffffffu, nib, 1);
        if ((tid & 1) == 0) grp[jj * kCb + (tid >> 1)] = static_cast<uint8_t>(nib | (up << 4));
    }
    if (tid == 0) *reinterpret_cast<float *>(grp + gh * kCb + 4 * jj) = step;
    if (jj == 0 && tid < kSummGroup - gh)                   // padding words after the steps
        *reinterpret_cast<uint32_t *>(grp + gh * kCb + 4 * (gh + tid)) = 0u;
}

// The exact sum, in token order, of one dimension of a page's 16 bf16 keys
// (bit patterns in the low 16 bits of v[t]), when their exponents allow it:
//  * a key is sig * 2^(e - 134) with an integer significand sig < 256 (e = the
//    exponent field, 1 for subnormals).  When the nonzero keys' exponents span
//    at most 40, every partial sum is an integer multiple of 2^(emin - 134)
//    below 2^52 in magnitude, so the sequential fp64 sum is exact and equals
//    the 64-bit integer sum of the significands shifted to the smallest
//    exponent: returns true with that sum in `acc` and emin in `emin`
//    (acc == 0 when every key is +-0 or they cancel: the fp64 sum is +0);
//  * wider spreads, infinities and NaNs return false.
__device__ __forceinline__ bool page_dim_sum_fixed(const uint32_t (&v)[kPageSize], long long &acc, int &emin_out)
{
    int emax = -1, emin = 1 << 30;
    bool special = false;
#pragma unroll
    for (int t = 0; t < kPageSize; ++t) {
        const int e = static_cast<int>((v[t] >> 7) & 0xFFu);
        special |= e == 0xFF;
        if (v[t] & 0x7FFFu) {                           // nonzero
            const int es = e > 0 ? e : 1;
            emax = max(emax, es);
            emin = min(emin, es);
        }
    }
    acc = 0;
    emin_out = 1;
    if (emax < 0) return true;                          // every key is +-0: 0 + ... = +0
    if (special || emax - emin > 40) return false;
#pragma unroll
    for (int t = 0; t < kPageSize; ++t) {
        const int e = static_cast<int>((v[t] >> 7) & 0xFFu);
        const long long sig = static_cast<long long>((v[t] & 0x7Fu) | (e > 0 ? 0x80u : 0u));
        const long long term = sig << max((e > 0 ? e : 1) - emin, 0);     // zeros: sig 0
        acc += (v[t] & 0x8000u) ? -term : term;
    }
    emin_out = emin;
    return true;
}

// The fp64 sum of the same keys in token order, starting from +0.
__device__ __forceinline__ double page_dim_sum_f64(const uint32_t (&v)[kPageSize])
{
    double sum = 0.0;
#pragma unroll
    for (int t = 0; t < kPageSize; ++t) sum += static_cast<double>(__uint_as_float(v[t] << 16));
    return sum;
}

// The fp64 sum of one dimension's 16 keys in token order, bit-exact (the
// integer form where it applies, fp64 adds otherwise).
__device__ __forceinline__ double page_dim_sum(const uint32_t (&v)[kPageSize])
{
    long long acc;
    int emin;
    if (page_dim_sum_fixed(v, acc, emin)) return ldexp(static_cast<double>(acc), emin - 134);
    return page_dim_sum_f64(v);
}

// acc * 2^e2 (|acc| < 2^62, finite and within the bf16 range once rounded)
// rounded to the nearest bf16, ties to even, by integer arithmetic.  The
// result's last place is 2^(e_lead - 7) for a leading bit of weight
// 2^e_lead >= 2^-126, else the subnormal step 2^-133; q, the rounded
// significand on that place, then gives the encoding as
// ((place + 133) << 7) + q for both kinds, a carry to q = 256 included.
__device__ __forceinline__ uint32_t fixed_to_bf16_rne(long long acc, int e2)
{
    if (acc == 0) return 0u;                            // an exact sum of 0 is +0
    const uint32_t sign = acc < 0 ? 0x8000u : 0u;
    const unsigned long long m =
        acc < 0 ? 0ull - static_cast<unsigned long long>(acc) : static_cast<unsigned long long>(acc);
    const int e_lead = 63 - __clzll(static_cast<long long>(m)) + e2;
    const int place = max(e_lead - 7, -133);
    const int sh = place - e2;                          // bits of m below the result's last place
    unsigned long long q;
    if (sh <= 0) {
        q = m << (-sh);
    } else {
        q = m >> sh;
        const unsigned long long rem = m & ((1ull << sh) - 1ull), half = 1ull << (sh - 1);
        q += (rem > half || (rem == half && (q & 1ull))) ? 1ull : 0ull;
    }
    return sign | (static_cast<uint32_t>(place + 133) << 7) + static_cast<uint32_t>(q);
}

// The low-bit record of KV head j from the warp's 128 fp64 means (lane l holds
// dimensions 4l .. 4l+3); the same quantiser as store_lowbit.
template <int kBits>
__device__ void store_lowbit_warp(const double (&mean)[4], uint8_t *rec, int j, int hkv)
{
    constexpr int kCb = lowbit_code_bytes(kBits);
    constexpr double kHalf = static_cast<double>(1 << (kBits - 1));
    const int lane = threadIdx.x & 31;
    bool bad = false;
    double a = 0.0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        bad |= !isfinite(mean[i]);
        a = fmax(a, fabs(mean[i]));
    }
    if (bad) a = 0.0;
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmax(a, __shfl_xor_sync(0xffffffffu, a, o));
    const bool any_bad = __any_sync(0xffffffffu, bad);
    const float step = any_bad ? 0.f : __double2float_rn(a / (kHalf - 0.5));
    int c[4] = {0, 0, 0, 0};
    if (step > 0.f) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            c[i] = static_cast<int>(fmin(fmax(floor(mean[i] / static_cast<double>(step)), -kHalf), kHalf - 1.0));
    }
    const int gh = lowbit_group_heads(hkv), jj = j % gh;
    uint8_t *grp = rec + (j / gh) * lowbit_group_bytes(kBits, hkv);
    if constexpr (kBits == 8) {
        *reinterpret_cast<uint32_t *>(grp + jj * kCb + 4 * lane) =
            static_cast<uint32_t>(c[0] & 0xFF) | (static_cast<uint32_t>(c[1] & 0xFF) << 8) |
            (static_cast<uint32_t>(c[2] & 0xFF) << 16) | (static_cast<uint32_t>(c[3] & 0xFF) << 24);
    } else {
        // element i sits in bits 2*(i%4) of byte i/4: the lane's 4 elements are byte `lane`
        grp[jj * kCb + lane] = static_cast<uint8_t>((c[0] + 2) | ((c[1] + 2) << 2) | ((c[2] + 2) << 4) |
                                                    ((c[3] + 2) << 6));
    }
    if (lane == 0) *reinterpret_cast<float *>(grp + gh * kCb + 4 * jj) = step;
    if (jj == 0 && lane < kSummGroup - gh)                  // padding words after the steps
        *reinterpret_cast<uint32_t *>(grp + gh * kCb + 4 * (gh + lane)) = 0u;
}

// One warp per (listed page, KV head), 8 per block: lane l loads 8 bytes
// (dimensions 4l .. 4l+3) of each of the 16 token rows, all 16 loads in
// flight, and forms the 4 means exactly (page_dim_sum).
constexpr int kSumWarps = 8;

template <int kFmt>
__global__ void __launch_bounds__(kSumWarps * 32, 3) k_summarize(const uint2 *__restrict__ k_pool,
                                                               uint8_t *__restrict__ summ,
                                                               const int32_t *__restrict__ phys_pages, int items,
                                                               int hkv, long long num_pages, uint32_t *status)
{
    const int item = blockIdx.x * kSumWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (item >= items) return;                               // warp-uniform
    const int j = item % hkv;
    const int p = phys_pages[item / hkv];
    if (p < 0 || p >= num_pages) {
        if (lane == 0 && status != nullptr) raise_status(status, kDevBadPage);
        return;
    }
    const size_t blk = static_cast<size_t>(p) * hkv + j;
    const uint2 *src = k_pool + blk * (kPageSize * kHeadDim / 4) + lane;
    uint2 row[kPageSize];
#pragma unroll
    for (int t = 0; t < kPageSize; ++t) row[t] = __ldg(src + t * (kHeadDim / 4));
    if constexpr (kFmt == kSummBf16) {
        // exponent fields of the lane's 4 dimensions (16-bit halves of the two
        // words), smallest and largest over the 16 tokens
        uint32_t mn[2] = {0xFFFFFFFFu, 0xFFFFFFFFu}, mx[2] = {0u, 0u};
#pragma unroll
        for (int t = 0; t < kPageSize; ++t) {
            const uint32_t ex = row[t].x & 0x7F807F80u, ey = row[t].y & 0x7F807F80u;
            mn[0] = __vminu2(mn[0], ex);
            mx[0] = __vmaxu2(mx[0], ex);
            mn[1] = __vminu2(mn[1], ey);
            mx[1] = __vmaxu2(mx[1], ey);
        }
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int sh = 16 * (i & 1);
            const uint32_t lo = (mn[i >> 1] >> sh) & 0xFFFFu, hi = (mx[i >> 1] >> sh) & 0xFFFFu;
            // every key normal (exponent field >= 1, so no zeros either), the
            // largest below 2^124 (16 of them stay below the fp32 limit) and a
            // span of at most 12: every fp32 partial sum is exact
            if (lo >= (1u << 7) && hi <= (250u << 7) && hi - lo <= (12u << 7)) {
                float sum = 0.f;
#pragma unroll
                for (int t = 0; t < kPageSize; ++t) {
                    const uint32_t w = i < 2 ? row[t].x : row[t].y;
                    sum += __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
                }
                out[i] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(sum * (1.f / kPageSize))));
            } else {
                uint32_t v[kPageSize];
#pragma unroll
                for (int t = 0; t < kPageSize; ++t) v[t] = ((i < 2 ? row[t].x : row[t].y) >> sh) & 0xFFFFu;
                long long acc;
                int emin;
                out[i] = page_dim_sum_fixed(v, acc, emin)
                             ? fixed_to_bf16_rne(acc, emin - 134 - 4)
                             : f64_to_bf16_rne(page_dim_sum_f64(v) * (1.0 / kPageSize));
            }
        }
        reinterpret_cast<uint2 *>(summ)[blk * (kHeadDim / 4) + lane] =
            make_uint2(out[0] | (out[1] << 16), out[2] | (out[3] << 16));
    } else {
        double mean[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t v[kPageSize];
#pragma unroll
            for (int t = 0; t < kPageSize; ++t) v[t] = ((i < 2 ? row[t].x : row[t].y) >> (16 * (i & 1))) & 0xFFFFu;
            mean[i] = page_dim_sum(v) * (1.0 / kPageSize);
        }
        store_lowbit_warp<summ_bits(kFmt)>(mean, summ + static_cast<size_t>(p) * summ_page_bytes(kFmt, hkv), j,
                                           hkv);
    }
}

// Append one token per request to a paged pool (one block per (request, KV
// head); 64 threads, two dimensions each).  The token of request r is token
// seq_lens[r] - 1: slot (L-1) % S of logical page (L-1) / S.  When that slot
// is the page's last, the page has just filled and its summary is computed
// here: the 15 earlier keys are read back from the pool, the new one is
// still in registers, and the mean is formed (fp64 in token order, which
// page_dim_sum reproduces exactly) and stored as k_summarize stores it.
__global__ void __launch_bounds__(64) k_append(const uint32_t *__restrict__ k_new,
                                               const uint32_t *__restrict__ v_new,
                                               uint32_t *__restrict__ k_pool, uint32_t *__restrict__ v_pool,
                                               uint8_t *__restrict__ summ,
                                               const int32_t *__restrict__ page_table,
                                               const int32_t *__restrict__ seq_lens, int hkv,
                                               int max_pages, long long num_pages, int fmt)
{
    const int r = blockIdx.x / hkv, j = blockIdx.x % hkv;
    const int L = seq_lens[r];
    if (L <= 0 || L > max_pages * kPageSize) return;       // nothing to append / out of range
    const int pos = L - 1, lp = pos / kPageSize, slot = pos % kPageSize;
    const int p = page_table[static_cast<size_t>(r) * max_pages + lp];
    if (p < 0 || p >= num_pages) return;
    const size_t blk = static_cast<size_t>(p) * hkv + j;
    const size_t src = (static_cast<size_t>(r) * hkv + j) * (kHeadDim / 2) + threadIdx.x;
    const uint32_t kn = k_new[src], vn = v_new[src];
    uint32_t *kb = k_pool + blk * (kPageSize * kHeadDim / 2) + threadIdx.x;
    kb[slot * (kHeadDim / 2)] = kn;
    v_pool[blk * (kPageSize * kHeadDim / 2) + slot * (kHeadDim / 2) + threadIdx.x] = vn;
    if (slot == kPageSize - 1) {
        double lo = 0.0, hi = 0.0;
#pragma unroll
        for (int t = 0; t < kPageSize - 1; ++t) {
            const uint32_t v = kb[t * (kHeadDim / 2)];
            lo += static_cast<double>(bf16_lo(v));
            hi += static_cast<double>(bf16_hi(v));
        }
        lo += static_cast<double>(bf16_lo(kn));
        hi += static_cast<double>(bf16_hi(kn));
        lo *= 1.0 / kPageSize;
        hi *= 1.0 / kPageSize;
        uint8_t *rec = summ + static_cast<size_t>(p) * summ_page_bytes(fmt, hkv);
        if (fmt == kSummQ8) {
            store_lowbit<8>(lo, hi, rec, j, hkv);
        } else if (fmt == kSummQ2) {
            store_lowbit<2>(lo, hi, rec, j, hkv);
        } else {
            reinterpret_cast<uint32_t *>(summ)[blk * (kHeadDim / 2) + threadIdx.x] =
                f64_to_bf16_rne(lo) | (f64_to_bf16_rne(hi) << 16);
        }
    }
}

cudaError_t launch_append(const void *k_new, const void *v_new, void *k_pool, void *v_pool,
                          void *summ, const int32_t *page_table, const int32_t *seq_lens,
                          int batch, int hkv, int max_pages, long long num_pages, int fmt,
                          cudaStream_t stream)
{
    k_append<<<static_cast<unsigned>(batch) * hkv, 64, 0, stream>>>(
        static_cast<const uint32_t *>(k_new), static_cast<const uint32_t *>(v_new),
        static_cast<uint32_t *>(k_pool), static_cast<uint32_t *>(v_pool),
        static_cast<uint8_t *>(summ), page_table, seq_lens, hkv, max_pages, num_pages, fmt);
    return cudaGetLastError();
}

cudaError_t launch_summarize(const void *k_pool, void *summ, const int32_t *phys_pages, int n,
                             int hkv, long long num_pages, int fmt, uint32_t *status,
                             cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    const int items = n * hkv;
    const unsigned grid = static_cast<unsigned>((items + kSumWarps - 1) / kSumWarps);
    const uint2 *kp = static_cast<const uint2 *>(k_pool);
    uint8_t *sm = static_cast<uint8_t *>(summ);
    if (fmt == kSummQ8)
        k_summarize<kSummQ8><<<grid, kSumWarps * 32, 0, stream>>>(kp, sm, phys_pages, items, hkv, num_pages, status);
    else if (fmt == kSummQ2)
        k_summarize<kSummQ2><<<grid, kSumWarps * 32, 0, stream>>>(kp, sm, phys_pages, items, hkv, num_pages, status);
    else
        k_summarize<kSummBf16><<<grid, kSumWarps * 32, 0, stream>>>(kp, sm, phys_pages, items, hkv, num_pages, status);
    return cudaGetLastError();
}

}  // namespace moira
