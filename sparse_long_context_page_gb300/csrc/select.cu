// The gamma-coverage selection of "MOIRA: Mass-Oriented Indexing with Ragged
// Attention for Long-Context Decoding", abstract: for every request, layer,
// KV head and step, keep the smallest set of pages whose estimated attention
// mass reaches gamma.
//
// Two kernels per layer:
//  k_score  : all SMs stream the page summaries once (16-byte loads, the G
//             query rows of a KV head sharing each load) and write the
//             log2-domain page logits plus per-chunk (max, sum 2^(s-max)).
//  k_select : one 1024-thread block per (request, KV head).  It merges the
//             chunk normalisers, forms m_p = (1/G) sum_h softmax_p(s_hp),
//             finds the cut mass by a radix descent over the fp32 bit
//             patterns (mass histograms kept as 2^-31 fixed-point integer
//             sums in native 32-bit shared atomics, so the result does not
//             depend on atomic order), then compacts the kept pages in
//             ascending logical order.
// Top-p over pages needs the global softmax and a cumulative sum ("Faster
// Flash Decoding", section 1 and figure 1); the histogram descent replaces a
// full sort.
#include "moira_device.cuh"
#include "moira_launch.h"

namespace moira {

// ---------------------------------------------------------------------------
// k_score
// ---------------------------------------------------------------------------
constexpr int kScoreThreads = 256;        // 8 warps
constexpr int kScoreItemsPerLane = 8;     // 32 pages * Hkv(<= 8) / 32 items per pass

// Lane layout: 8 lanes per (page, KV head) item, 16 dimensions (32 bytes) per
// lane; 4 items per warp and 32 per block pass.  Because 32 is a multiple of
// Hkv, a lane always serves the same KV head and keeps that head's G=4 query
// slices (64 floats) in registers for the whole block.
__global__ void __launch_bounds__(kScoreThreads, 2) k_score(
    const uint16_t *__restrict__ q, const uint16_t *__restrict__ summ,
    const int32_t *__restrict__ page_table, const int32_t *__restrict__ seq_lens, int hq, int hkv,
    int max_pages, long long num_pages, float scale_log2, float *__restrict__ scores,
    float *__restrict__ chunks, int n_chunks, uint32_t *status)
{
    __shared__ float s_s[32 * kScoreChunk];   // [Hq <= 32][32 pages]
    pdl_trigger();
    pdl_wait();                               // q and the score buffers follow earlier kernels
    const int r = blockIdx.y;
    const int chunk = blockIdx.x;
    int L = seq_lens[r];
    L = L < 0 ? 0 : (L > max_pages * kPageSize ? max_pages * kPageSize : L);
    const int F = L / kPageSize;
    const int p0 = chunk * kScoreChunk;
    if (p0 >= F) return;
    const int np = min(kScoreChunk, F - p0);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane & 7;
    const int j = (warp * 4 + (lane >> 3)) % hkv;

    float qr[kGroup][16];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
        const uint4 *qp = reinterpret_cast<const uint4 *>(
            q + (static_cast<size_t>(r) * hq + j * kGroup + g) * kHeadDim + sub * 16);
        const uint4 a = __ldg(qp), b = __ldg(qp + 1);
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            qr[g][2 * i] = bf16_lo(w[i]);
            qr[g][2 * i + 1] = bf16_hi(w[i]);
        }
    }

    const int n_items = np * hkv;
    const int32_t *row = page_table + static_cast<size_t>(r) * max_pages + p0;
    // two passes of 4 items per lane: 4 x 32 B loads in flight per lane
#pragma unroll
    for (int k0 = 0; k0 < kScoreItemsPerLane; k0 += 4) {
        if (warp * 4 + 32 * k0 >= n_items) break;            // warp-uniform
        uint4 buf[4][2];
        bool bad[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int it = warp * 4 + (lane >> 3) + 32 * (k0 + k);
            bad[k] = false;
            buf[k][0] = buf[k][1] = make_uint4(0, 0, 0, 0);
            if (it < n_items) {
                const int phys = __ldg(row + it / hkv);
                if (phys < 0 || phys >= num_pages) {
                    bad[k] = true;
                } else {
                    const uint4 *sp = reinterpret_cast<const uint4 *>(
                        summ + (static_cast<size_t>(phys) * hkv + j) * kHeadDim + sub * 16);
                    buf[k][0] = __ldg(sp);
                    buf[k][1] = __ldg(sp + 1);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int it = warp * 4 + (lane >> 3) + 32 * (k0 + k);
            if (warp * 4 + 32 * (k0 + k) >= n_items) break;  // warp-uniform
            const uint32_t w[8] = {buf[k][0].x, buf[k][0].y, buf[k][0].z, buf[k][0].w,
                                   buf[k][1].x, buf[k][1].y, buf[k][1].z, buf[k][1].w};
            float dot[kGroup];
#pragma unroll
            for (int g = 0; g < kGroup; ++g) dot[g] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float x0 = bf16_lo(w[i]), x1 = bf16_hi(w[i]);
#pragma unroll
                for (int g = 0; g < kGroup; ++g)
                    dot[g] = fmaf(qr[g][2 * i + 1], x1, fmaf(qr[g][2 * i], x0, dot[g]));
            }
#pragma unroll
            for (int g = 0; g < kGroup; ++g) {
                dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 1);
                dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 2);
                dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], 4);
            }
            if (sub == 0 && it < n_items) {
                const int pl = it / hkv;
                if (bad[k]) raise_status(status, kDevBadPage);
#pragma unroll
                for (int g = 0; g < kGroup; ++g) {
                    const int h = j * kGroup + g;
                    const float sv = bad[k] ? -INFINITY : dot[g] * scale_log2;
                    s_s[h * kScoreChunk + pl] = sv;
                    scores[(static_cast<size_t>(r) * hq + h) * max_pages + p0 + pl] = sv;
                }
            }
        }
    }
    __syncthreads();
    // per-head (max, sum 2^(s - max)) over this chunk
    for (int h = warp; h < hq; h += kScoreThreads / 32) {
        const float v = lane < np ? s_s[h * kScoreChunk + lane] : -INFINITY;
        float mx = v;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float e = (lane < np && mx != -INFINITY) ? exp2f(v - mx) : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
        if (lane == 0) {
            float *c = chunks + ((static_cast<size_t>(r) * hq + h) * n_chunks + chunk) * 2;
            c[0] = mx;
            c[1] = e;
        }
    }
}

// ---------------------------------------------------------------------------
// k_select
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
// Level-1 bins: the fp32 bit pattern >> 16 (exponent + 7 fraction bits, 128
// bins per octave) for masses in [2^-32, 2); bin 0 gathers everything below.
constexpr uint32_t kKeyLo = 95u << 7;
constexpr int kL1Bins = (16384 - static_cast<int>(kKeyLo)) + 1;     // 4225
constexpr int kL1PerThread = (kL1Bins + kSelThreads - 1) / kSelThreads;   // 5
constexpr int kL2Bins = 256;

__device__ __forceinline__ int l1_bin(uint32_t x)
{
    const uint32_t k = x >> 16;
    return k < kKeyLo ? 0 : static_cast<int>(k - kKeyLo) + 1;
}
__device__ __forceinline__ uint32_t l1_lo(int b) { return b == 0 ? 0u : (static_cast<uint32_t>(b - 1) + kKeyLo) << 16; }
__device__ __forceinline__ uint32_t l1_hi(int b) { return b == 0 ? (kKeyLo << 16) : (static_cast<uint32_t>(b) + kKeyLo) << 16; }

// Mass as a 2^-31 fixed-point integer.  Masses sum to 1 (to fp32 rounding),
// so every histogram bin and every partial sum fits in 32 bits; rounding each
// mass costs at most 2^-32, i.e. < 1e-5 over 32768 pages.
__device__ __forceinline__ uint32_t to_fx(uint32_t x)
{
    return __float2uint_rn(__uint_as_float(x) * 0x1p31f);
}

// Exclusive scan over the block in thread order; *total gets the sum.
__device__ unsigned long long block_excl_scan(unsigned long long v, unsigned long long *s_warp,
                                              unsigned long long *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        unsigned long long w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    const unsigned long long off = warp > 0 ? s_warp[warp - 1] : 0ull;
    *total = s_warp[kSelWarps - 1];
    __syncthreads();
    return off + x - v;
}

struct SelectShared {
    uint32_t h1[kL1Bins];
    uint32_t h2[kL2Bins];
    unsigned long long scan[32];
    unsigned long long above;
    uint32_t lo, hi;
    int found;
    int kept;
    float mmax[kGroup];
    float wgt[kGroup];
};

__global__ void __launch_bounds__(kSelThreads) k_select(
    const float *__restrict__ scores, const float *__restrict__ chunks,
    const int32_t *__restrict__ page_table, const int32_t *__restrict__ seq_lens, int hq, int hkv,
    int max_pages, int n_chunks, long long num_pages, unsigned long long gamma_fx, int dense,
    int32_t *__restrict__ lists, int32_t *__restrict__ lengths, uint32_t *status)
{
    extern __shared__ __align__(16) uint32_t s_bits[];       // [max_pages] mass bit patterns
    __shared__ SelectShared sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_trigger();
    pdl_wait();                               // scores and chunk stats come from k_score
    const int u = blockIdx.x;
    const int r = u / hkv, j = u % hkv;
    int L = seq_lens[r];
    if (L < 0 || L > max_pages * kPageSize) {
        if (tid == 0) raise_status(status, kDevBadLen);
        L = L < 0 ? 0 : max_pages * kPageSize;
    }
    const int F = L / kPageSize, T = (L % kPageSize) != 0;
    const int32_t *row = page_table + static_cast<size_t>(r) * max_pages;
    int32_t *out = lists + static_cast<size_t>(u) * max_pages;

    if (dense || F == 0) {                         // every page, no estimate
        for (int p = tid; p < F + T; p += kSelThreads) out[p] = row[p];
        if (tid == 0) lengths[u] = F + T;
        return;
    }

    // 1. merge the chunk normalisers of the group's G heads
    const int nch = (F + kScoreChunk - 1) / kScoreChunk;
    if (warp < kGroup) {
        const float *c = chunks + (static_cast<size_t>(r) * hq + j * kGroup + warp) * n_chunks * 2;
        float mx = -INFINITY;
        for (int i = lane; i < nch; i += 32) mx = fmaxf(mx, c[2 * i]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float z = 0.f;
        if (mx != -INFINITY)
            for (int i = lane; i < nch; i += 32)
                if (c[2 * i] != -INFINITY) z += c[2 * i + 1] * exp2f(c[2 * i] - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        if (lane == 0) {
            sh.mmax[warp] = mx == -INFINITY ? 0.f : mx;
            sh.wgt[warp] = z > 0.f ? 1.f / (kGroup * z) : 0.f;
        }
    }
    for (int b = tid; b < kL1Bins; b += kSelThreads) sh.h1[b] = 0u;
    if (tid == 0) { sh.found = 0; sh.above = 0ull; }
    __syncthreads();

    // 2. masses and the level-1 histogram (logits of 8 pages per thread are
    //    loaded together before any arithmetic)
    const float *sc = scores + (static_cast<size_t>(r) * hq + j * kGroup) * max_pages;
    float mm[kGroup], ww[kGroup];
#pragma unroll
    for (int g = 0; g < kGroup; ++g) {
        mm[g] = sh.mmax[g];
        ww[g] = sh.wgt[g];
    }
    for (int p0 = 0; p0 < F; p0 += 8 * kSelThreads) {
        float v[8][kGroup];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int p = p0 + k * kSelThreads + tid;
#pragma unroll
            for (int g = 0; g < kGroup; ++g)
                v[k][g] = p < F ? __ldcg(sc + static_cast<size_t>(g) * max_pages + p) : -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int p = p0 + k * kSelThreads + tid;
            if (p < F) {
                float m = 0.f;
#pragma unroll
                for (int g = 0; g < kGroup; ++g) m += exp2f(v[k][g] - mm[g]) * ww[g];
                m = fminf(fmaxf(m, 0.f), 1.5f);        // NaN -> 0
                const uint32_t x = __float_as_uint(m);
                s_bits[p] = x;
                atomicAdd(&sh.h1[l1_bin(x)], to_fx(x));
            }
        }
    }
    __syncthreads();

    // 3. level-1 cut: thread t owns bins (hi_t .. lo_t] counted from the top
    {
        const int top = kL1Bins - 1 - tid * kL1PerThread;
        unsigned long long mine = 0ull;
#pragma unroll
        for (int i = 0; i < kL1PerThread; ++i)
            if (top - i >= 0) mine += sh.h1[top - i];
        unsigned long long total;
        unsigned long long acc = block_excl_scan(mine, sh.scan, &total);
        if (acc < gamma_fx && acc + mine >= gamma_fx) {
#pragma unroll
            for (int i = 0; i < kL1PerThread; ++i) {
                const int b = top - i;
                if (b < 0) break;
                if (acc + sh.h1[b] >= gamma_fx) {
                    sh.lo = l1_lo(b);
                    sh.hi = l1_hi(b);
                    sh.above = acc;
                    sh.found = 1;
                    break;
                }
                acc += sh.h1[b];
            }
        }
    }
    __syncthreads();

    // 4. refine inside [lo, hi) with 256-bin passes until one bit pattern is
    //    left (at most 4 passes: 30 bits of range, 8 bits per pass)
    for (int pass = 0; sh.found && sh.hi - sh.lo > 1u; ++pass) {
        if (pass >= 6) {                                // cannot happen: exact integer sums
            if (tid == 0) raise_status(status, kDevBadLen);
            break;
        }
        const uint32_t lo = sh.lo, hi = sh.hi;
        const uint32_t width = hi - lo;
        const int bits = 32 - __clz(width - 1u);
        const int shift = bits > 8 ? bits - 8 : 0;
        const int nb = static_cast<int>((width - 1u) >> shift) + 1;
        if (tid < kL2Bins) sh.h2[tid] = 0u;
        __syncthreads();
        for (int p = tid; p < F; p += kSelThreads) {
            const uint32_t x = s_bits[p];
            if (x >= lo && x < hi) atomicAdd(&sh.h2[(x - lo) >> shift], to_fx(x));
        }
        __syncthreads();
        if (warp == 0) {
            // lane owns bins [top-7, top] with top = nb-1-8*lane, walked downwards
            const int top = nb - 1 - 8 * lane;
            unsigned long long mine = 0ull;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (top - i >= 0) mine += sh.h2[top - i];
            unsigned long long x = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            unsigned long long acc = sh.above + x - mine;
            const unsigned long long need = gamma_fx;
            if (acc < need && acc + mine >= need) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int b = top - i;
                    if (b < 0) break;
                    if (acc + sh.h2[b] >= need) {
                        const uint32_t nlo = lo + (static_cast<uint32_t>(b) << shift);
                        const uint32_t span = 1u << shift;
                        sh.lo = nlo;
                        sh.hi = (hi - nlo < span) ? hi : nlo + span;
                        sh.above = acc;
                        break;
                    }
                    acc += sh.h2[b];
                }
            }
        }
        __syncthreads();
    }

    // 5. cut value and how many pages tied at it are needed
    uint32_t cut;
    unsigned long long need_tied;
    if (sh.found) {
        cut = sh.lo;
        const unsigned long long cfx = to_fx(cut);
        const unsigned long long rest = gamma_fx - sh.above;     // > 0
        need_tied = (rest + cfx - 1ull) / cfx;                    // cfx > 0: it carried the crossing
    } else {                                                      // total < gamma: keep all
        cut = 0u;
        need_tied = 0xFFFFFFFFull;
    }

    // 6. ordered compaction: thread t owns a contiguous run of pages; the
    //    physical ids of the first 8 are fetched before the scan
    const int ept = (F + kSelThreads - 1) / kSelThreads;
    const int pb = min(F, tid * ept), pe = min(F, pb + ept);
    int32_t pref[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) pref[k] = (pb + k < pe) ? __ldg(row + pb + k) : 0;
    uint32_t gt = 0, eq = 0;
    for (int p = pb; p < pe; ++p) {
        const uint32_t x = s_bits[p];
        gt += x > cut;
        eq += x == cut;
    }
    unsigned long long total;
    const unsigned long long pre = block_excl_scan(gt | (static_cast<unsigned long long>(eq) << 32),
                                                   sh.scan, &total);
    const uint32_t gt_pre = static_cast<uint32_t>(pre), eq_pre = static_cast<uint32_t>(pre >> 32);
    unsigned long long eq_run = eq_pre;
    int pos = static_cast<int>(gt_pre + (eq_pre < need_tied ? eq_pre : need_tied));
    bool badp = false;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int p = pb + k;
        if (p < pe) {
            const uint32_t x = s_bits[p];
            bool keep = x > cut;
            if (x == cut) {
                keep = eq_run < need_tied;
                ++eq_run;
            }
            if (keep) {
                badp |= (pref[k] < 0 || pref[k] >= num_pages);
                out[pos++] = pref[k];
            }
        }
    }
    for (int p = pb + 8; p < pe; ++p) {
        const uint32_t x = s_bits[p];
        bool keep = x > cut;
        if (x == cut) {
            keep = eq_run < need_tied;
            ++eq_run;
        }
        if (keep) {
            const int32_t phys = row[p];
            badp |= (phys < 0 || phys >= num_pages);
            out[pos++] = phys;
        }
    }
    if (badp) raise_status(status, kDevBadPage);
    if (tid == 0) {
        const unsigned long long gt_all = total & 0xFFFFFFFFull, eq_all = total >> 32;
        const int kept = static_cast<int>(gt_all + (eq_all < need_tied ? eq_all : need_tied));
        if (T) out[kept] = row[F];
        lengths[u] = kept + T;
    }
}

// ---------------------------------------------------------------------------
cudaError_t launch_score(const void *q, const void *summ, const int32_t *page_table,
                         const int32_t *seq_lens, int batch, int hq, int hkv, int max_pages,
                         long long num_pages, float scale_log2, float *scores, float *chunks,
                         uint32_t *status, cudaStream_t stream)
{
    const int n_chunks = (max_pages + kScoreChunk - 1) / kScoreChunk;
    dim3 grid(n_chunks, batch);
    return launch_pdl(k_score, grid, dim3(kScoreThreads), 0, stream,
                      static_cast<const uint16_t *>(q), static_cast<const uint16_t *>(summ),
                      page_table, seq_lens, hq, hkv, max_pages, num_pages, scale_log2, scores,
                      chunks, n_chunks, status);
}

cudaError_t launch_select(const float *scores, const float *chunks, const int32_t *page_table,
                          const int32_t *seq_lens, int batch, int hq, int hkv, int max_pages,
                          long long num_pages, unsigned long long gamma_fx, bool dense,
                          int32_t *lists, int32_t *lengths, uint32_t *status, cudaStream_t stream)
{
    const int n_chunks = (max_pages + kScoreChunk - 1) / kScoreChunk;
    const size_t smem = dense ? 0 : sizeof(uint32_t) * static_cast<size_t>(max_pages);
    if (!dense) {
        cudaError_t e = cudaFuncSetAttribute(k_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(k_select, dim3(batch * hkv), dim3(kSelThreads), smem, stream, scores, chunks,
                      page_table, seq_lens, hq, hkv, max_pages, n_chunks, num_pages, gamma_fx,
                      dense ? 1 : 0, lists, lengths, status);
}

}  // namespace moira
