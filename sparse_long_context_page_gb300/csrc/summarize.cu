// Page summaries: the bf16 mean key of every (page, KV head) block.
//
// "MOIRA: Mass-Oriented Indexing with Ragged Attention for Long-Context
// Decoding", abstract: the coverage rule works on an *estimated* attention
// mass per page, which needs per-page metadata.  The form used here is the
// mean vector of the page's keys, one of the block summaries named in
// "Faster Flash Decoding", section 2 (related work).
//
// The 16 keys are summed in fp64 (exact for bf16 inputs of moderate range)
// and the mean is rounded once to bf16, ties to even.  This runs when a page
// fills, outside the decode step, so fp64 throughput does not matter here.
//
// Low-bit formats store the same fp64 mean in 8 or 2 bits per element with
// the symmetric mid-rise quantiser that "Faster Flash Decoding", section 3.1,
// uses for its low-bit key thumbnails: one fp32 step per (page, KV head),
//   step = max_i |mean_i| / (2^(bits-1) - 1/2)   (fp64, rounded once to fp32)
//   code = floor(mean_i / step), clamped to [-2^(bits-1), 2^(bits-1) - 1]
// standing for (code + 1/2) * step; no zero level, so signs survive.  A
// non-finite mean element, a zero mean or a step that rounds to 0 gives
// step 0 and codes 0.
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

// fp64 sums over the page's 16 tokens of this thread's two dimensions
// (2*tid, 2*tid+1), in token order; `src` points at the thread's word of
// token 0.
__device__ __forceinline__ void token_sums(const uint32_t *src, double &lo, double &hi)
{
    lo = 0.0;
    hi = 0.0;
#pragma unroll
    for (int t = 0; t < kPageSize; ++t) {
        const uint32_t v = __ldg(src + t * (kHeadDim / 2));
        lo += static_cast<double>(bf16_lo(v));
        hi += static_cast<double>(bf16_hi(v));
    }
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

// One block per (listed page, KV head); 64 threads, two dimensions each.
__global__ void __launch_bounds__(64) k_summarize(const uint32_t *__restrict__ k_pool,
                                                  uint32_t *__restrict__ summ,
                                                  const int32_t *__restrict__ phys_pages, int hkv,
                                                  long long num_pages, uint32_t *status)
{
    const int item = blockIdx.x;
    const int j = item % hkv;
    const int idx = item / hkv;
    const int p = phys_pages[idx];
    if (p < 0 || p >= num_pages) {
        if (threadIdx.x == 0 && status != nullptr) raise_status(status, kDevBadPage);
        return;
    }
    const size_t blk = (static_cast<size_t>(p) * hkv + j);
    double lo, hi;
    token_sums(k_pool + blk * (kPageSize * kHeadDim / 2) + threadIdx.x, lo, hi);
    const uint32_t blo = f64_to_bf16_rne(lo * (1.0 / kPageSize));
    const uint32_t bhi = f64_to_bf16_rne(hi * (1.0 / kPageSize));
    summ[blk * (kHeadDim / 2) + threadIdx.x] = blo | (bhi << 16);
}

// Low-bit summaries: one block per (listed page, KV head), 64 threads.
template <int kBits>
__global__ void __launch_bounds__(64) k_summarize_lowbit(const uint32_t *__restrict__ k_pool,
                                                         uint8_t *__restrict__ summ,
                                                         const int32_t *__restrict__ phys_pages,
                                                         int hkv, long long num_pages, int rec_bytes)
{
    const int item = blockIdx.x;
    const int j = item % hkv;
    const int p = phys_pages[item / hkv];
    if (p < 0 || p >= num_pages) return;                     // block-uniform
    double lo, hi;
    token_sums(k_pool + (static_cast<size_t>(p) * hkv + j) * (kPageSize * kHeadDim / 2) + threadIdx.x,
               lo, hi);
    store_lowbit<kBits>(lo * (1.0 / kPageSize), hi * (1.0 / kPageSize),
                        summ + static_cast<size_t>(p) * rec_bytes, j, hkv);
}

// Append one token per request to a paged pool (one block per (request, KV
// head); 64 threads, two dimensions each).  The token of request r is token
// seq_lens[r] - 1: slot (L-1) % S of logical page (L-1) / S.  When that slot
// is the page's last, the page has just filled and its summary is computed
// here: the 15 earlier keys are read back from the pool, the new one is
// still in registers, and the mean is formed and stored as in k_summarize
// (or k_summarize_lowbit, by `fmt`).
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
    const unsigned grid = static_cast<unsigned>(n) * hkv;
    const uint32_t *kp = static_cast<const uint32_t *>(k_pool);
    if (fmt == kSummQ8)
        k_summarize_lowbit<8><<<grid, 64, 0, stream>>>(kp, static_cast<uint8_t *>(summ), phys_pages,
                                                       hkv, num_pages, summ_page_bytes(fmt, hkv));
    else if (fmt == kSummQ2)
        k_summarize_lowbit<2><<<grid, 64, 0, stream>>>(kp, static_cast<uint8_t *>(summ), phys_pages,
                                                       hkv, num_pages, summ_page_bytes(fmt, hkv));
    else
        k_summarize<<<grid, 64, 0, stream>>>(kp, static_cast<uint32_t *>(summ), phys_pages, hkv,
                                             num_pages, status);
    return cudaGetLastError();
}

}  // namespace moira
