// The gamma-coverage selection of "MOIRA: Mass-Oriented Indexing with Ragged
// Attention for Long-Context Decoding", abstract: per request, layer and KV
// head at each decode step, pick the fewest pages whose estimated share of
// the attention adds up to gamma.
//
// Two kernels per layer:
//  k_score  : all SMs stream the page summaries once (bulk copies into shared
//             memory; blocks of 32 pages x 4 KV heads) and compute the page
//             logits on the tensor cores, the G query rows of a KV head
//             sharing every summary.  Per chunk of 32
//             pages and query head it stores the chunk max M_c and sum
//             Z_c = sum_p 2^(s_p - M_c), and per page the chunk-relative
//             weight e_p = 2^(s_p - M_c) (log2-domain logits).
//  k_select : one 1024-thread block per (request, KV head).  It bulk-copies
//             the group's weights and chunk statistics into shared memory,
//             merges the normalisers, forms
//                 m_p = (1/G) sum_h e_hp 2^(M_hc - M_h) / Z_h
//                     = (1/G) sum_h softmax_p(s_h.)
//             and finds the cut mass by a radix descent over the fp32 bit
//             patterns (mass histograms kept as 2^-31 fixed-point integer sums
//             in native 32-bit shared atomics, so the result does not depend
//             on atomic order), then compacts the kept pages in ascending
//             logical order with warp ballots.
// Top-p over pages needs the global softmax and a cumulative sum ("Faster
// Flash Decoding", section 1 and figure 1); the histogram descent replaces a
// full sort.
#include "select_core.cuh"

namespace moira {

// ---------------------------------------------------------------------------
// k_score
// ---------------------------------------------------------------------------
constexpr int kScoreConsumers = 8;        // warps: one (KV head, 16-page half) of an item each
constexpr int kScoreThreads = (kScoreConsumers + 1) * 32;   // + one producer warp
constexpr int kScoreHeads = 4;            // KV heads per item
constexpr int kScoreMaxStages = 4;
static_assert(kScoreHeads * 2 <= kScoreConsumers, "one (KV head, 16-page half) per consumer warp");
static_assert(kScoreHeads == kSummGroup, "a score item reads one low-bit head group");

__device__ __forceinline__ void score_consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kScoreConsumers * 32) : "memory");
}

// Per query head of an item: chunk max, chunk sum and the chunk-relative
// weights from the item's logits s_s[local head][page] (log2 domain, -inf
// for pages that do not count); 8 lanes per head (4 pages each), 4 heads
// per warp instruction, consumer warps only.
__device__ __forceinline__ void score_chunk_stats(const float *s_s, int nh, int jb, int r, int chunk,
                                                  int p0, int hq, int ld, int ldc,
                                                  float *__restrict__ weights,
                                                  float *__restrict__ chunks)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hql = nh * kGroup;
    for (int h0 = warp * 4; h0 < hql; h0 += 4 * kScoreConsumers) {
        const int hl = h0 + (lane >> 3);
        const int sub = lane & 7;
        float4 v = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        if (hl < hql) v = *reinterpret_cast<const float4 *>(&s_s[hl * kScoreChunk + sub * 4]);
        float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        const float ms = mx == -INFINITY ? 0.f : mx;
        const float4 e = make_float4(exp2f(v.x - ms), exp2f(v.y - ms), exp2f(v.z - ms), exp2f(v.w - ms));
        float sum = (e.x + e.y) + (e.z + e.w);
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        if (hl < hql) {
            const int h = jb * kGroup + hl;
            float *dst = weights + (static_cast<size_t>(r) * hq + h) * ld + p0 + sub * 4;
            *reinterpret_cast<float4 *>(dst) = e;          // pages past F are never read
            if (sub == 0) {
                float *c = chunks + (static_cast<size_t>(r) * hq + h) * ldc + chunk * 2;
                *reinterpret_cast<float2 *>(c) = make_float2(mx, sum);
            }
        }
    }
}

// fp16 pair {lo, hi} (lo in the low half) from two floats, rounded to nearest.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two 8-bit codes as an exact fp16 pair: byte u = c + 128 placed under the
// exponent of 1024 reads as 1024 + u, and 1024 + u - 1152 = c.  `sel` picks
// bytes 0,1 (0x5140) or 2,3 (0x5342) of the biased word.
__device__ __forceinline__ uint32_t q8_pair(uint32_t biased, uint32_t sel)
{
    return hsub2(__byte_perm(biased, 0x64646464u, sel), 0x64806480u);
}

// Two 2-bit codes (stored as c + 2 at bits 0-1 and 16-17 of v) as an exact
// fp16 pair: 1024 + u - 1026 = c.
__device__ __forceinline__ uint32_t q2_pair(uint32_t v)
{
    return hsub2((v & 0x00030003u) | 0x64006400u, 0x64026402u);
}

// Shared-memory stride of one page slot for low-bit summaries: the page's
// head group (codes and steps), padded so that the lanes of one load phase
// (8 lanes of 16-byte loads for Q8, 16 lanes of 8-byte loads for Q2) hit
// distinct banks.
__host__ __device__ constexpr int score_lowbit_stride(int bits, int hkv)
{
    return (lowbit_group_bytes(bits, hkv) + 127) / 128 * 128 + (bits == 8 ? 16 : 32);
}

// Shared-memory stride of one page slot, by summary format: bf16 rows are
// padded by 16 bytes so that the 8 ldmatrix rows of consecutive pages fall
// in different banks; low-bit slots as score_lowbit_stride.
__host__ __device__ constexpr int score_stride(int fmt, int nh, int hkv)
{
    return fmt == kSummBf16 ? nh * kHeadDim * 2 + 16 : score_lowbit_stride(summ_bits(fmt), hkv);
}

// Position of a score work item: request r, slice of nh KV heads, chunk of
// 32 full pages.  In the persistent walk `nck` is the request's chunk count
// (only chunks holding full pages are visited).
struct ScoreCursor {
    int r, slice, chunk, nck;
};

// Items of request r in the persistent walk: n_slices * ceil(F_r / 32).
__device__ __forceinline__ int score_items_of(int L, int max_pages, int n_slices)
{
    L = L < 0 ? 0 : (L > max_pages * kPageSize ? max_pages * kPageSize : L);
    return n_slices * ((L / kPageSize + kScoreChunk - 1) / kScoreChunk);
}

// Cursor of item g of the persistent walk (s_pref: exclusive prefix of the
// requests' item counts, s_pref[batch] = total).
__device__ __forceinline__ ScoreCursor score_cursor_at(int g, const int *s_pref, int batch, int n_slices)
{
    int lo = 0, hi = batch;                   // the last r with s_pref[r] <= g (never an empty request)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_pref[mid] <= g) lo = mid;
        else hi = mid;
    }
    ScoreCursor c;
    c.r = lo;
    c.nck = (s_pref[lo + 1] - s_pref[lo]) / n_slices;
    const int local = g - s_pref[lo];
    c.slice = local / c.nck;
    c.chunk = local % c.nck;
    return c;
}

__device__ __forceinline__ void score_cursor_next(ScoreCursor &c, const int *s_pref, int batch, int n_slices)
{
    if (++c.chunk < c.nck) return;
    c.chunk = 0;
    if (++c.slice < n_slices) return;
    c.slice = 0;
    do {
        ++c.r;
    } while (c.r < batch - 1 && s_pref[c.r + 1] == s_pref[c.r]);
    if (c.r < batch) c.nck = (s_pref[c.r + 1] - s_pref[c.r]) / n_slices;
}

// Page logits of every (request, KV head, full page) and their per-chunk
// softmax statistics.  A work item is (request, slice of kScoreHeads KV
// heads, chunk of 32 consecutive full pages).
//
// Warp-specialised: the producer warp brings each valid page's summaries for
// the item's heads into a shared-memory stage by 1-D bulk copies
// (cp.async.bulk) on the stage's "full" mbarrier; the 8 consumer warps take
// one (KV head, 16-page half) each, compute the logits on the tensor cores
// and the chunk statistics, and free the stage on its "empty" mbarrier.
// Two launch shapes (template argument kPersistent):
//  * single wave: one block per item of the full
//    (request, slice, chunk) grid, one stage; blocks past a request's full
//    pages exit.  Page ids, the sequence length and the query fragments are
//    all requested before the summaries are waited for;
//  * persistent: a grid of resident blocks.  Every block
//    scans the sequence lengths (exclusive prefix of the requests' item
//    counts in shared memory), takes an equal range of the non-empty items
//    in (request, slice, chunk) order and runs a ring of `stages` stages;
//    the producer requests the next item's page ids while it issues the
//    current copies, and consumers request the query fragments before
//    waiting for the data.
//
// Logits, for KV head j and 16 pages: S^T[h][p] = sum_d q_{4j+h}[d] kbar_p[d]
// by mma.m16n8k16 with A = the group's 4 query rows (repeated in rows 4-7):
//  * bf16 summaries: B = the summary rows via ldmatrix, bf16 operands;
//  * low-bit summaries (value = (c + 1/2) * step): fp16 operands.  A code c
//    becomes an exact fp16 by placing its biased bits under the exponent of
//    1024 and subtracting (a byte permute or mask and one f16x2 subtract per
//    two codes); each query head is scaled by 2^k so that its largest element
//    lies in [2^14, 2^15), which keeps its bf16 values exact in fp16; the 1/2
//    of every level returns in the epilogue:
//      s_p = step_p * (2^-k sum_i (2^k q_i) c_i + (1/2) sum_i q_i).
//    Lane t of a quad holds elements 32t .. 32t+31 of its page (a 32-byte run
//    for Q8, 8 bytes for Q2) and the contraction index is permuted so that
//    every fp16 pair forms in place (Q8: 32t + 4s + {0,1} and {2,3} at k-step
//    s; Q2: 32t + {s, s+8} and 32t + {16+s, 24+s}), the query fragments
//    taking the same permutation.
template <int kFmt, bool kPersistent>
__global__ void __launch_bounds__(kScoreThreads, kPersistent ? 3 : 4) k_score(
    const uint16_t *__restrict__ q, const uint8_t *__restrict__ summ,
    const int32_t *__restrict__ page_table, const int32_t *__restrict__ seq_lens, int batch, int hq,
    int hkv, int max_pages, int ld, long long num_pages, float scale_log2,
    float *__restrict__ weights, float *__restrict__ chunks, int ldc, int stages, int early,
    uint32_t *status)
{
    constexpr bool kLow = kFmt != kSummBf16;
    constexpr int kBits = summ_bits(kFmt);
    constexpr int kCb = kLow ? lowbit_code_bytes(kBits) : kHeadDim * 2;   // code bytes per head
    extern __shared__ __align__(128) uint8_t s_score[];       // [stages][32 pages][stride], s_pref
    __shared__ __align__(16) float s_s[kScoreHeads * kGroup * kScoreChunk];  // [local q head][page]
    __shared__ uint32_t s_ok[kScoreMaxStages];               // per stage: pages loaded
    __shared__ int s_wsum[kScoreConsumers + 1];
    __shared__ __align__(8) unsigned long long s_full[kScoreMaxStages], s_empty[kScoreMaxStages];
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const WaitGuard wg{&s_abort, status};
    const int nh = min(hkv, kScoreHeads);
    const int n_slices = hkv / nh;
    const int n_chunks = (max_pages + kScoreChunk - 1) / kScoreChunk;
    const uint32_t stride = static_cast<uint32_t>(score_stride(kFmt, nh, hkv));
    const uint32_t code_bytes = static_cast<uint32_t>(nh) * kCb;
    // bytes of one page that an item copies: its heads' bf16 rows, or its
    // low-bit head group (codes, steps, padding)
    const uint32_t copy_bytes = kLow ? static_cast<uint32_t>(lowbit_group_bytes(kBits, hkv)) : code_bytes;
    const size_t rec = static_cast<size_t>(summ_page_bytes(kFmt, hkv));
    int *s_pref = reinterpret_cast<int *>(s_score + static_cast<size_t>(stages) * kScoreChunk * stride);
    if (tid == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(smem_u32(&s_full[s]), 1);
            mbar_init(smem_u32(&s_empty[s]), 1);
        }
        mbar_fence_init();
        guard_init(wg);
    }
    // q and the score buffers follow earlier kernels, so they are touched only
    // after the wait.  With `early`, the launch follows this library's
    // attention kernel in the same step (which writes neither the page table,
    // the lengths nor the summaries, all of which the step's first scoring
    // launch has waited for), so the plan, the page ids and the first items'
    // summary copies go out before it.  Every thread triggers its dependents
    // after its own wait: k_select relies on that.
    if (!early) {
        pdl_wait();
        pdl_trigger();
    }

    // ---- the block's items ------------------------------------------------------
    int g0, g1;                               // item range (fewer than 2^21 items)
    ScoreCursor c0;
    if constexpr (kPersistent) {
        const int per = (batch + kScoreThreads - 1) / kScoreThreads;
        const int rb = min(batch, tid * per), re = min(batch, rb + per);
        int mine = 0;
        for (int r = rb; r < re; ++r) mine += score_items_of(__ldg(seq_lens + r), max_pages, n_slices);
        int x = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        int run = x - mine;
        for (int w = 0; w < warp; ++w) run += s_wsum[w];
        for (int r = rb; r < re; ++r) {
            s_pref[r] = run;
            run += score_items_of(__ldg(seq_lens + r), max_pages, n_slices);
        }
        if (tid == kScoreThreads - 1) s_pref[batch] = run;
        __syncthreads();
        const long long W = s_pref[batch];
        g0 = static_cast<int>(blockIdx.x * W / gridDim.x);
        g1 = static_cast<int>((blockIdx.x + 1) * W / gridDim.x);
        if (g0 < g1) c0 = score_cursor_at(g0, s_pref, batch, n_slices);
    } else {
        __syncthreads();                      // barriers initialised
        g0 = 0;
        g1 = 1;
        c0.chunk = blockIdx.x % n_chunks;
        c0.slice = (blockIdx.x / n_chunks) % n_slices;
        c0.r = blockIdx.x / (n_chunks * n_slices);
        c0.nck = n_chunks;
    }
    if (g0 >= g1) return;                     // block-uniform

    if (warp == kScoreConsumers) {
        // ---- producer ----------------------------------------------------------
        const uint64_t pol = l2_evict_first();    // summaries are read once per step
        ScoreCursor c = c0;
        int L = __ldg(seq_lens + c.r);
        int phys = c.chunk * kScoreChunk + lane < max_pages
                       ? __ldg(page_table + static_cast<size_t>(c.r) * max_pages + c.chunk * kScoreChunk + lane)
                       : -1;
        // With `early`, the summaries are read before the wait too: the kernel
        // before this one is the previous layer's attention, which writes no
        // summaries, so the copies of the first ring's worth of items land
        // while it finishes.  The producer waits (and only then triggers the
        // dependents) once the ring is full or its items are issued.
        bool waited = !early;
        for (int g = g0; g < g1; ++g) {
            // next item's page ids and length, requested before this item's copies
            ScoreCursor n = c;
            int L_n = L, phys_n = -1;
            if (g + 1 < g1) {
                score_cursor_next(n, s_pref, batch, n_slices);
                if (n.r != c.r) L_n = __ldg(seq_lens + n.r);
                if (n.chunk * kScoreChunk + lane < max_pages)
                    phys_n = __ldg(page_table + static_cast<size_t>(n.r) * max_pages + n.chunk * kScoreChunk + lane);
            }
            const int Lc = L < 0 ? 0 : (L > max_pages * kPageSize ? max_pages * kPageSize : L);
            const int np = min(kScoreChunk, Lc / kPageSize - c.chunk * kScoreChunk);
            if (np <= 0) break;               // single wave: past the request's full pages
            const bool ok = lane < np && phys >= 0 && phys < num_pages;
            const uint32_t okm = __ballot_sync(0xffffffffu, ok);
            if (lane < np && !ok && c.slice == 0) raise_status(status, kDevBadPage);
            const int it = g - g0;
            const int stage = it % stages;
            const uint32_t use = static_cast<uint32_t>(it / stages);
            if (use > 0) mbar_wait_g(smem_u32(&s_empty[stage]), (use - 1) & 1u, wg);
            const uint32_t full = smem_u32(&s_full[stage]);
            if (lane == 0) {
                s_ok[stage] = okm;
                mbar_arrive_expect_tx(full, __popc(okm) * copy_bytes);
            }
            __syncwarp();
            if (ok) {
                bulk_load_hint(smem_u32(s_score + (static_cast<uint32_t>(stage) * kScoreChunk + lane) * stride),
                               summ + static_cast<size_t>(phys) * rec + static_cast<size_t>(c.slice) * copy_bytes,
                               copy_bytes, full, pol);
            }
            c = n;
            L = L_n;
            phys = phys_n;
            if (!waited && (g - g0 + 1 == stages || g + 1 == g1)) {
                pdl_wait();
                pdl_trigger();
                waited = true;
            }
        }
        if (!waited) {                        // the items ran out early (single wave)
            pdl_wait();
            pdl_trigger();
        }
        return;
    }

    // ---- consumers -------------------------------------------------------------
    if (early) {
        pdl_wait();
        pdl_trigger();
    }
    const int hrow = (lane >> 2) & 3;
    const int t = lane & 3;
    const bool has_item = warp < nh * 2;      // warp-uniform
    const int jl = warp >> 1, half = warp & 1;
    ScoreCursor c = c0;
    // query fragments of the current (request, slice); consecutive items of a
    // block mostly share them, so they are fetched (and, for low-bit
    // summaries, scaled and packed to fp16) only when (request, slice) changes
    uint32_t qw[16];
    float down = 1.f, half_qsum = 0.f;
    int q_r = -1, q_slice = -1;
    for (int g = g0; g < g1; ++g) {
        const int jb = c.slice * nh;
        if (has_item && (c.r != q_r || c.slice != q_slice)) {
            q_r = c.r;
            q_slice = c.slice;
            const uint16_t *qrow = q + (static_cast<size_t>(c.r) * hq + (jb + jl) * kGroup + hrow) * kHeadDim;
            if constexpr (!kLow) {
                const uint16_t *qa = qrow + 2 * t;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    qw[2 * ks] = __ldg(reinterpret_cast<const uint32_t *>(qa + ks * 16));
                    qw[2 * ks + 1] = __ldg(reinterpret_cast<const uint32_t *>(qa + ks * 16 + 8));
                }
            } else {
                // the lane's 32 query elements 32t .. 32t+31 as bf16 pairs
                const uint4 *qv4 = reinterpret_cast<const uint4 *>(qrow + 32 * t);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 v = __ldg(qv4 + i);
                    qw[4 * i] = v.x;
                    qw[4 * i + 1] = v.y;
                    qw[4 * i + 2] = v.z;
                    qw[4 * i + 3] = v.w;
                }
                float qmax = 0.f, qsum = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float lo = bf16_lo(qw[i]), hi = bf16_hi(qw[i]);
                    qmax = fmaxf(qmax, fmaxf(fabsf(lo), fabsf(hi)));
                    qsum += lo + hi;
                }
                qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
                qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
                qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
                qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
                int k = 0;
                if (qmax > 0.f)
                    k = min(max(14 - (static_cast<int>((__float_as_uint(qmax) >> 23) & 0xFFu) - 127), -126), 126);
                const float up = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
                down = __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
                half_qsum = 0.5f * qsum;
                // fp16 query fragments, packed in place.  Q8: qw[2s], qw[2s+1]
                // hold elements 4s + {0,1}, {2,3} (k-step s).  Q2: k-step s
                // takes elements {s, s+8} and {16+s, 24+s}, built from the
                // pairs (2j, 2j+1) and (8+2j, 9+2j): even s sits in qw[s/2] and
                // qw[8 + s/2], odd s in qw[4 + s/2] and qw[12 + s/2].
                if constexpr (kBits == 8) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) qw[i] = pack_f16x2(bf16_lo(qw[i]) * up, bf16_hi(qw[i]) * up);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int o = 0; o < 16; o += 8) {
                            const uint32_t x = qw[o + j], y = qw[o + 4 + j];
                            qw[o + j] = pack_f16x2(bf16_lo(x) * up, bf16_lo(y) * up);
                            qw[o + 4 + j] = pack_f16x2(bf16_hi(x) * up, bf16_hi(y) * up);
                        }
                    }
                }
            }
        }
        if constexpr (!kPersistent) {         // single wave: is this item inside the request?
            int L = __ldg(seq_lens + c.r);
            L = L < 0 ? 0 : (L > max_pages * kPageSize ? max_pages * kPageSize : L);
            if (c.chunk * kScoreChunk >= L / kPageSize) return;     // block-uniform
        }
        const int it = g - g0;
        const int stage = it % stages;
        const uint32_t use = static_cast<uint32_t>(it / stages);
        mbar_wait_g(smem_u32(&s_full[stage]), use & 1u, wg);
        const uint32_t okm = s_ok[stage];
        const uint8_t *base = s_score + static_cast<uint32_t>(stage) * kScoreChunk * stride;
        if (has_item) {
            float acc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            if constexpr (!kLow) {
                // ldmatrix rows: (pages 0-7, dims +0), (0-7, +8), (8-15, +0), (8-15, +8)
                const int prow = half * 16 + (lane & 7) + ((lane >> 4) << 3);
                const uint32_t rbase = smem_u32(base) + prow * stride + jl * kCb + (((lane >> 3) & 1) << 4);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(rbase + ks * 32, b0, b1, b2, b3);
                    mma_bf16_16816(acc[0], qw[2 * ks], 0u, qw[2 * ks + 1], 0u, b0, b1);
                    mma_bf16_16816(acc[1], qw[2 * ks], 0u, qw[2 * ks + 1], 0u, b2, b3);
                }
            } else {
                auto a0 = [&](int ks) { return kBits == 8 ? qw[2 * ks] : qw[(ks & 1) * 4 + (ks >> 1)]; };
                auto a1 = [&](int ks) { return kBits == 8 ? qw[2 * ks + 1] : qw[8 + (ks & 1) * 4 + (ks >> 1)]; };
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint8_t *src = base + (half * 16 + nt * 8 + (lane >> 2)) * stride + jl * kCb + t * (kCb / 4);
                    if constexpr (kBits == 8) {
                        const uint4 x0 = *reinterpret_cast<const uint4 *>(src);
                        const uint4 x1 = *reinterpret_cast<const uint4 *>(src + 16);
                        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {
                            const uint32_t u = w[ks] ^ 0x80808080u;
                            mma_f16_16816(acc[nt], a0(ks), 0u, a1(ks), 0u, q8_pair(u, 0x5140u),
                                          q8_pair(u, 0x5342u));
                        }
                    } else {
                        const uint2 x = *reinterpret_cast<const uint2 *>(src);
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            mma_f16_16816(acc[nt], a0(ks), 0u, a1(ks), 0u, q2_pair(x.x >> (2 * ks)),
                                          q2_pair(x.y >> (2 * ks)));
                    }
                }
            }
            if (lane < 16) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int pl = half * 16 + nt * 8 + 2 * t;
                    const int hl = jl * kGroup + hrow;
                    float s0, s1;
                    if constexpr (kLow) {
                        const float st0 = reinterpret_cast<const float *>(base + pl * stride + code_bytes)[jl];
                        const float st1 = reinterpret_cast<const float *>(base + (pl + 1) * stride + code_bytes)[jl];
                        s0 = fmaf(acc[nt][0], down, half_qsum) * st0 * scale_log2;
                        s1 = fmaf(acc[nt][1], down, half_qsum) * st1 * scale_log2;
                    } else {
                        s0 = acc[nt][0] * scale_log2;
                        s1 = acc[nt][1] * scale_log2;
                    }
                    if (!((okm >> pl) & 1u)) s0 = -INFINITY;
                    if (!((okm >> (pl + 1)) & 1u)) s1 = -INFINITY;
                    *reinterpret_cast<float2 *>(&s_s[hl * kScoreChunk + pl]) = make_float2(s0, s1);
                }
            }
        }
        score_consumer_bar();                 // the stage is read and the logits are complete
        if (tid == 0) mbar_arrive(smem_u32(&s_empty[stage]));
        score_chunk_stats(s_s, nh, jb, c.r, c.chunk, c.chunk * kScoreChunk, hq, ld, ldc, weights, chunks);
        score_consumer_bar();                 // s_s is free again
        if (g + 1 < g1) score_cursor_next(c, s_pref, batch, n_slices);
    }
    // after a give-up, let the copies still in flight land before the block
    // exits (their landing is what the skipped waits were for)
    if (tid == 0 && guard_failed(wg)) {
        const uint64_t deadline = globaltimer() + kDrainLimitNs;
        const int N = g1 - g0;
        for (int s = 0; s < stages && s < N; ++s) {
            const int last = N - 1 - ((N - 1 - s) % stages);          // last item on stage s
            mbar_drain(smem_u32(&s_full[s]), static_cast<uint32_t>(last / stages) & 1u, deadline);
        }
    }
}

// ---------------------------------------------------------------------------
// k_select
// ---------------------------------------------------------------------------
constexpr int kSelThreads = 1024;
constexpr int kSelWarps = kSelThreads / 32;
// Stripes of 1024 pages: 8 up to 8192 pages per request, 16 up to 16384
// (the kernel is instantiated for both; registers hold one value per stripe).
constexpr int kSelStripesMax = kMaxPagesPerSeq / kSelThreads;
static_assert(kSelStripesMax % 4 == 0, "masses: 4 pages per thread per pass");
constexpr int kL1PerThread = (kL1Bins + kSelThreads - 1) / kSelThreads;   // 5
// Exclusive scan over the block in thread order; *total gets the sum.
__device__ unsigned long long sel_excl_scan(unsigned long long v, unsigned long long *s_warp,
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

static_assert(kPairMax * 4 <= kSelThreads, "pairwise path: at least 4 threads per candidate");
static_assert(kMaxPagesPerSeq / kScoreChunk <= 2 * 256, "normalisers: at most two chunks per thread and head");

struct SelectShared {
    uint32_t h1[kL1Bins];
    uint32_t h2[kL2Bins];
    uint32_t cand[kCand];                   // mass bits of the crossing bin's pages
    uint32_t cand_fx[kPairMax];             // their fixed-point masses (pairwise path only)
    uint16_t cand_idx[kCand];               // their page indices (pairwise path only)
    int ncand;
    unsigned long long scan[32];
    unsigned long long above;
    uint32_t cnt[kSelStripesMax * kSelWarps];           // (stripe, warp): gt | eq << 16
    uint32_t cnt_total;
    uint32_t lo, hi;
    int found;
    float red[kSelWarps];
    float red2[kSelWarps];
    float mmax[kGroup];
    float zinv[kGroup];
    uint32_t xmax;                          // largest mass pattern (top-delta)
};

// Dynamic shared memory of k_select: per-chunk factors and the mass bit
// patterns (the weights and chunk statistics are read from L2, where k_score
// has just written them).
__host__ __device__ inline size_t select_smem_bytes(int max_pages, int ldc)
{
    const size_t wld = static_cast<size_t>(weights_ld(max_pages));
    return sizeof(float4) * static_cast<size_t>(ldc / 2) + sizeof(uint32_t) * wld;
}

template <int kSelStripes>
__global__ void __launch_bounds__(kSelThreads) k_select(
    const float *__restrict__ weights, const float *__restrict__ chunks,
    const int32_t *__restrict__ page_table, const int32_t *__restrict__ seq_lens, int hq, int hkv,
    int max_pages, int ld, int ldc, long long num_pages, int rule, unsigned long long target,
    float delta, int dense,
    int32_t *__restrict__ lists, int32_t *__restrict__ lengths, uint32_t *status)
{
    extern __shared__ __align__(16) float s_dyn[];
    __shared__ SelectShared sh;
    float4 *s_f = reinterpret_cast<float4 *>(s_dyn);               // [ldc/2] per-chunk factors
    uint32_t *s_bits = reinterpret_cast<uint32_t *>(s_f + ldc / 2);   // [ld] mass bits

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Before the wait: reads of the caller's inputs (page table, lengths) and
    // shared-memory set-up.  With gamma < 1 this block can only have started
    // once k_score passed its own wait (k_score signals its dependents after
    // it), so the kernels that wrote those inputs have finished.  A dense
    // launch has no k_score before it and waits first.
    if (dense) pdl_wait();
    const int u = blockIdx.x;
    const int r = u / hkv, j = u % hkv;
    const int32_t *row = page_table + static_cast<size_t>(r) * max_pages;
    int32_t *out = lists + static_cast<size_t>(u) * max_pages;
    int L = seq_lens[r];
    // page ids of this thread's pages (page k*1024 + tid) in flight early
    int32_t pref[kSelStripes];
#pragma unroll
    for (int k = 0; k < kSelStripes; ++k) {
        const int p = k * kSelThreads + tid;
        pref[k] = p < max_pages ? __ldg(row + p) : 0;
    }
    const int32_t tail_pre = (tid == 0 && L > 0 && L <= max_pages * kPageSize && (L % kPageSize) != 0)
                                 ? __ldg(row + L / kPageSize) : 0;
    if (L < 0 || L > max_pages * kPageSize) {
        if (tid == 0) raise_status(status, kDevBadLen);
        L = L < 0 ? 0 : max_pages * kPageSize;
    }
    const int F = L / kPageSize, T = (L % kPageSize) != 0;
    for (int b = tid; b < kL1Bins; b += kSelThreads) sh.h1[b] = 0u;
    if (tid == 0) {
        sh.found = 0;
        sh.above = 0ull;
        sh.xmax = 0u;
    }
    pdl_trigger();
    pdl_wait();                               // weights and chunk stats come from k_score;
                                              // lists may still be read by the last attention
    if (rule == kRuleTopK && target == 0ull && F > 0 && !dense) {   // no full page, only the tail
        if (tid == 0) {
            if (T) out[0] = row[F];
            lengths[u] = T;
        }
        return;
    }
    if (dense || F == 0 || (rule == kRuleTopK && target >= static_cast<unsigned long long>(F))) {
        // every page, no estimate
        for (int p = tid; p < F + T; p += kSelThreads) out[p] = row[p];
        if (tid == 0) lengths[u] = F + T;
        return;
    }
    const int nch = (F + kScoreChunk - 1) / kScoreChunk;
    const int nstripes = (F + kSelThreads - 1) / kSelThreads;

    // 1. the group's weight rows and chunk statistics are in L2 (k_score
    //    wrote them): the first pass of weights is requested now, so that its
    //    latency overlaps the normalisers
    const float *wrow = weights + (static_cast<size_t>(r) * hq + j * kGroup) * ld;
    float4 wpre[kGroup];
    {
        const int p = tid * 4;
#pragma unroll
        for (int h = 0; h < kGroup; ++h)
            wpre[h] = p < F ? __ldg(reinterpret_cast<const float4 *>(wrow + h * ld + p))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // 2. normalisers of the group's heads.  Thread -> (head tid/256, chunks
    //    tid%256 + 256 i): M = max of the chunk maxima, e_c = 2^(M_c - M) once
    //    per chunk, Z = sum_c e_c Z_c; the chunk factor is e_c / (G Z).
    {
        // thread -> (head tid/256, chunks tid%256 and tid%256 + 256): warp w of
        // a head is its virtual warp w of the fixed-order reduction
        const int hg = tid >> 8, ci = tid & 255;
        const float *crow = chunks + (static_cast<size_t>(r) * hq + j * kGroup + hg) * ldc;
        float cm[2] = {-INFINITY, -INFINITY}, cz[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kSelStripes / 8; ++i) {
            const int c = ci + 256 * i;
            if (c < nch) {
                const float2 cs = __ldg(reinterpret_cast<const float2 *>(crow + 2 * c));
                cm[i] = cs.x;
                cz[i] = cs.y;
            }
        }
        const float mx = warp_max_butterfly(fmaxf(cm[0], cm[1]));
        if (lane == 0) sh.red[warp] = mx;
        __syncthreads();
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) M = fmaxf(M, sh.red[hg * 8 + w]);
        const float z = warp_sum_butterfly(chunk_weight_sum(cm[0], cz[0], cm[1], cz[1], M));
        if (lane == 0) sh.red2[warp] = z;
        __syncthreads();
        const float zinv = head_zinv(&sh.red2[hg * 8]);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            if (ci + 256 * i < nch)
                reinterpret_cast<float *>(s_f)[4 * (ci + 256 * i) + hg] = chunk_factor(cm[i], M, zinv);
    }
    __syncthreads();

    // 3. masses (natural page order, no exponentials) and the level-1
    //    histogram; thread t takes 4 consecutive pages per pass (one chunk
    //    factor, 16-byte loads and stores).  k_score writes whole 32-page
    //    chunks, so the 4 weights at p < F are all written.
#pragma unroll
    for (int k = 0; k < kSelStripes / 4; ++k) {
        const int p = (k * kSelThreads + tid) * 4;
        uint32_t xs[4] = {0u, 0u, 0u, 0u};
        if (p < F) {
            const float4 f = s_f[p / kScoreChunk];
            float4 w0, w1, w2, w3;
            if (k == 0) {
                w0 = wpre[0];
                w1 = wpre[1];
                w2 = wpre[2];
                w3 = wpre[3];
            } else {
                w0 = __ldg(reinterpret_cast<const float4 *>(wrow + p));
                w1 = __ldg(reinterpret_cast<const float4 *>(wrow + ld + p));
                w2 = __ldg(reinterpret_cast<const float4 *>(wrow + 2 * ld + p));
                w3 = __ldg(reinterpret_cast<const float4 *>(wrow + 3 * ld + p));
            }
            xs[0] = page_mass_bits(w0.x, w1.x, w2.x, w3.x, f);
            xs[1] = page_mass_bits(w0.y, w1.y, w2.y, w3.y, f);
            xs[2] = page_mass_bits(w0.z, w1.z, w2.z, w3.z, f);
            xs[3] = page_mass_bits(w0.w, w1.w, w2.w, w3.w, f);
            *reinterpret_cast<uint4 *>(s_bits + p) = make_uint4(xs[0], xs[1], xs[2], xs[3]);
        }
        if ((k * kSelThreads + warp * 32) * 4 < F) {        // warp-uniform: the warp has pages
            if (rule == kRuleTopDelta) {      // only the largest mass is needed
                uint32_t mx = 0u;
#pragma unroll
                for (int i = 0; i < 4; ++i) mx = max(mx, p + i < F ? xs[i] : 0u);
                mx = __reduce_max_sync(0xffffffffu, mx);
                if (lane == 0) atomicMax(&sh.xmax, mx);
            } else {
                // masses below 2^-32 are 0 in fixed point and add nothing to
                // the coverage histogram (most pages of a peaked group)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t w = rule_weight(rule, xs[i]);
                    hist_add_warp(sh.h1, static_cast<uint32_t>(l1_bin(xs[i])), w, p + i < F && w != 0u);
                }
            }
        }
    }
    __syncthreads();

    if (rule != kRuleTopDelta) {             // block-uniform: top-delta needs no descent
        // 4. level-1 cut: thread t owns bins (top_t - kL1PerThread, top_t] from the top
        {
            const int top = kL1Bins - 1 - tid * kL1PerThread;
            unsigned long long mine = 0ull;
    #pragma unroll
            for (int i = 0; i < kL1PerThread; ++i)
                if (top - i >= 0) mine += sh.h1[top - i];
            unsigned long long total;
            unsigned long long acc = sel_excl_scan(mine, sh.scan, &total);
            if (acc < target && acc + mine >= target) {
    #pragma unroll
                for (int i = 0; i < kL1PerThread; ++i) {
                    const int b = top - i;
                    if (b < 0) break;
                    if (acc + sh.h1[b] >= target) {
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

        // 5. refine inside [lo, hi) until one bit pattern is left.  The pages of
        //    the crossing bin are gathered first; when they fit in kCand (the
        //    usual case: a level-1 bin spans 1/128 of an octave) one warp refines
        //    them without block barriers, otherwise 256-bin passes run over all
        //    pages.  Both use the same integer sums, so the cut is identical.
        if (tid == 0) sh.ncand = 0;
        __syncthreads();
        if (sh.found) {
            // ballots first, one slot reservation per warp, then the writes
            const uint32_t lo = sh.lo, hi = sh.hi;
            uint32_t xk[kSelStripes];
            unsigned mk[kSelStripes];
            int cntw = 0;
    #pragma unroll
            for (int k = 0; k < kSelStripes; ++k) {
                const int p = k * kSelThreads + tid;
                xk[k] = p < F ? s_bits[p] : 0u;
                mk[k] = __ballot_sync(0xffffffffu, p < F && xk[k] >= lo && xk[k] < hi);
                cntw += __popc(mk[k]);
            }
            if (cntw) {                                          // warp-uniform
                int base = 0;
                if (lane == 0) base = atomicAdd(&sh.ncand, cntw);
                base = __shfl_sync(0xffffffffu, base, 0);
                const unsigned lt = (1u << lane) - 1u;
    #pragma unroll
                for (int k = 0; k < kSelStripes; ++k) {
                    if ((mk[k] >> lane) & 1u) {
                        const int slot = base + __popc(mk[k] & lt);
                        if (slot < kCand) {
                            sh.cand[slot] = xk[k];
                            sh.cand_idx[slot] = static_cast<uint16_t>(k * kSelThreads + tid);
                            if (slot < kPairMax) sh.cand_fx[slot] = rule_weight(rule, xk[k]);
                        }
                    }
                    base += __popc(mk[k]);
                }
            }
        }
        __syncthreads();
        const bool use_pair = sh.found && sh.ncand <= kPairMax;
        const bool use_cand = sh.found && !use_pair && sh.ncand <= kCand;
        if (use_pair) {
            // candidate c: masses ranked before it (larger, or equal with a lower
            // page index); the candidate whose running sum crosses gamma is the
            // cut.  2^lg threads (lanes of one warp) share a candidate's sums.
            const int nc = sh.ncand;
            const unsigned long long above0 = sh.above;
            __syncthreads();                                 // every thread has read `above`
            const int lg = nc <= 32 ? 5 : nc <= 64 ? 4 : nc <= 128 ? 3 : 2;
            const int ci = tid >> lg, part = tid & ((1 << lg) - 1);
            uint32_t gt_sum = 0u, tie_before = 0u;          // <= the total mass: fits 32 bits
            uint32_t x = 0u, xi = 0u;
            if (ci < nc) {
                x = sh.cand[ci];
                xi = sh.cand_idx[ci];
    #pragma unroll 4
                for (int c = part; c < nc; c += 1 << lg) {
                    const uint32_t y = sh.cand[c];
                    const uint32_t fy = sh.cand_fx[c];
                    gt_sum += y > x ? fy : 0u;
                    tie_before += (y == x && sh.cand_idx[c] < xi) ? fy : 0u;
                }
            }
            for (int o = 1; o < (1 << lg); o <<= 1) {
                gt_sum += __shfl_xor_sync(0xffffffffu, gt_sum, o);
                tie_before += __shfl_xor_sync(0xffffffffu, tie_before, o);
            }
            if (ci < nc && part == 0) {
                const unsigned long long before = above0 + gt_sum + tie_before;
                if (before < target && before + sh.cand_fx[ci] >= target) {   // exactly one candidate
                    sh.lo = x;
                    sh.hi = x + 1u;
                    sh.above = above0 + gt_sum;
                }
            }
            __syncthreads();
        } else if (use_cand) {
            if (warp == 0) {
                uint32_t lo = sh.lo, hi = sh.hi;
                unsigned long long above = sh.above;
                warp_refine(sh.cand, sh.ncand, sh.h2, rule, target, lo, hi, above);
                if (lane == 0) {
                    sh.lo = lo;
                    sh.hi = hi;
                    sh.above = above;
                    if (hi - lo > 1u) raise_status(status, kDevBadLen);
                }
            }
            __syncthreads();
        } else {
            for (int pass = 0; sh.found && sh.hi - sh.lo > 1u; ++pass) {
                if (pass >= 6) {                               // cannot happen: exact integer sums
                    if (tid == 0) raise_status(status, kDevBadLen);
                    break;
                }
                const uint32_t lo = sh.lo, hi = sh.hi;
                const uint32_t width = hi - lo;
                const int nbits = 32 - __clz(width - 1u);
                const int shift = nbits > 8 ? nbits - 8 : 0;
                const int nb = static_cast<int>((width - 1u) >> shift) + 1;
                if (tid < kL2Bins) sh.h2[tid] = 0u;
                __syncthreads();
    #pragma unroll
                for (int k = 0; k < kSelStripes; ++k) {
                    const int p = k * kSelThreads + tid;
                    if (k * kSelThreads >= F) break;              // warp-uniform
                    const uint32_t x = p < F ? s_bits[p] : 0u;
                    hist_add_warp(sh.h2, (x - lo) >> shift, rule_weight(rule, x), p < F && x >= lo && x < hi);
                }
                __syncthreads();
                if (warp == 0) {
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
                    if (acc < target && acc + mine >= target) {
    #pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int b = top - i;
                            if (b < 0) break;
                            if (acc + sh.h2[b] >= target) {
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
        }
    }

    // 6. cut value and how many pages tied at it are needed
    // (32-bit: gamma - above <= 2^31 and the cut's fixed-point mass < 2^32)
    uint32_t cut, need_tied;
    if (rule == kRuleTopDelta) {              // keep mass >= delta * max: every page at or above
        const float thr = fmaxf(delta * __uint_as_float(sh.xmax), 0.f);
        cut = __float_as_uint(thr);
        need_tied = 0xFFFFFFFFu;
    } else if (sh.found) {
        cut = sh.lo;
        const uint32_t cfx = rule_weight(rule, cut);               // > 0: it carried the crossing
        const uint32_t d = static_cast<uint32_t>(target - sh.above);
        need_tied = d / cfx + (d % cfx != 0u ? 1u : 0u);
    } else {                                                      // total < gamma: keep all
        cut = 0u;
        need_tied = 0xFFFFFFFFu;
    }

    // 7. ordered compaction by stripes of 1024 pages: per (stripe, warp) counts
    //    of pages above and at the cut (16 bits each: at most 8192), one warp
    //    scans them in page order, then warp ballots place the kept pages
    const unsigned lt_mask = (1u << lane) - 1u;
    unsigned gt_m[kSelStripes], eq_m[kSelStripes];
#pragma unroll
    for (int k = 0; k < kSelStripes; ++k) {
        gt_m[k] = eq_m[k] = 0u;
        if (k < nstripes) {
            const int p = k * kSelThreads + tid;
            const uint32_t x = p < F ? s_bits[p] : 0u;
            gt_m[k] = __ballot_sync(0xffffffffu, p < F && x > cut);
            eq_m[k] = __ballot_sync(0xffffffffu, p < F && x == cut);
            if (lane == 0) sh.cnt[k * kSelWarps + warp] = __popc(gt_m[k]) | (__popc(eq_m[k]) << 16);
        }
    }
    __syncthreads();
    if (warp == 0) {                          // lane l: entries S*l .. S*l+S-1 (S stripes)
        uint32_t v[kSelStripes], run = 0u;
#pragma unroll
        for (int i = 0; i < kSelStripes; ++i) {
            const int e = lane * kSelStripes + i;
            const uint32_t c = e < nstripes * kSelWarps ? sh.cnt[e] : 0u;
            v[i] = run;
            run += c;
        }
        uint32_t x = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        const uint32_t base = x - run;
#pragma unroll
        for (int i = 0; i < kSelStripes; ++i)
            if (lane * kSelStripes + i < nstripes * kSelWarps) sh.cnt[lane * kSelStripes + i] = base + v[i];
        if (lane == 31) sh.cnt_total = x;
    }
    __syncthreads();
    static_assert(kSelStripes * kSelWarps == 32 * kSelStripes, "one warp scans the compaction counts");
    bool badp = false;
#pragma unroll
    for (int k = 0; k < kSelStripes; ++k) {
        if (k < nstripes && (gt_m[k] | eq_m[k]) != 0u) {     // warp-uniform
            const uint32_t base = sh.cnt[k * kSelWarps + warp];
            const uint32_t gt_before = (base & 0xFFFFu) + __popc(gt_m[k] & lt_mask);
            const uint32_t eq_before = (base >> 16) + __popc(eq_m[k] & lt_mask);
            const bool is_gt = (gt_m[k] >> lane) & 1u, is_eq = (eq_m[k] >> lane) & 1u;
            if (is_gt || (is_eq && eq_before < need_tied)) {
                const int pos = static_cast<int>(gt_before + (eq_before < need_tied ? eq_before : need_tied));
                badp |= (pref[k] < 0 || pref[k] >= num_pages);
                out[pos] = pref[k];
            }
        }
    }
    if (badp) raise_status(status, kDevBadPage);
    if (tid == 0) {
        const uint32_t gt_all = sh.cnt_total & 0xFFFFu, eq_all = sh.cnt_total >> 16;
        const int kept = static_cast<int>(gt_all + (eq_all < need_tied ? eq_all : need_tied));
        if (T) out[kept] = tail_pre;
        lengths[u] = kept + T;
    }
}

// ---------------------------------------------------------------------------
// Per-device records of each score launch shape's shared-memory limit and
// single-wave capacity, at namespace scope with internal linkage (a static
// local of the function template below would be shared with any other
// library in the process that instantiates it).
namespace {
std::atomic<int> g_score_single_seen[3][64], g_score_single_fit[3][64][4], g_score_ring_seen[3][64];
}

template <int kFmt>
cudaError_t launch_score_fmt(const void *q, const void *summ, const int32_t *page_table,
                             const int32_t *seq_lens, int batch, int hq, int hkv, int max_pages,
                             long long num_pages, float scale_log2, float *weights, float *chunks,
                             bool early, uint32_t *status, cudaStream_t stream)
{
    // stages of the persistent ring: the low-bit formats take a deeper ring
    // in about the shared memory of bf16's two stages
    constexpr int kStagesMax = kFmt == kSummBf16 ? 2 : (kFmt == kSummQ8 ? 3 : kScoreMaxStages);
    static_assert(kStagesMax <= kScoreMaxStages, "stage ring");
    const int nh = hkv < kScoreHeads ? hkv : kScoreHeads;
    const long long n_items = static_cast<long long>(batch) * (hkv / nh) * ((max_pages + kScoreChunk - 1) / kScoreChunk);
    const size_t stage_bytes = static_cast<size_t>(kScoreChunk) * score_stride(kFmt, nh, hkv);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // single wave: one block per item with one stage, when every item fits
    // (resident blocks cached per (device, Hkv): they never change in a context)
    std::atomic<int> *single_seen = g_score_single_seen[kFmt];
    std::atomic<int>(*single_fit)[4] = g_score_single_fit[kFmt];
    const int hk = hkv == 1 ? 0 : (hkv == 2 ? 1 : (hkv == 4 ? 2 : 3));
    int fit = dev < 64 ? single_fit[dev][hk].load(std::memory_order_relaxed) : 0;
    if (fit == 0) {
        if ((e = raise_smem_limit(k_score<kFmt, false>, stage_bytes, single_seen)) != cudaSuccess) return e;
        int per_sm = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_score<kFmt, false>, kScoreThreads,
                                                               stage_bytes)) != cudaSuccess)
            return e;
        fit = sms * (per_sm > 0 ? per_sm : 1);
        if (dev < 64) single_fit[dev][hk].store(fit, std::memory_order_relaxed);
    }
    if (n_items <= fit)
        return launch_pdl(k_score<kFmt, false>, dim3(static_cast<unsigned>(n_items)), dim3(kScoreThreads),
                          stage_bytes, stream, static_cast<const uint16_t *>(q),
                          static_cast<const uint8_t *>(summ), page_table, seq_lens, batch, hq, hkv,
                          max_pages, weights_ld(max_pages), num_pages, scale_log2, weights, chunks,
                          chunks_ld(max_pages), 1, early ? 1 : 0, status);
    // persistent: resident blocks with the ring and the plan's prefix array
    std::atomic<int> *ring_seen = g_score_ring_seen[kFmt];
    const size_t smem = kStagesMax * stage_bytes + align_up(static_cast<size_t>(batch + 1) * 4, 16);
    if ((e = raise_smem_limit(k_score<kFmt, true>, smem, ring_seen)) != cudaSuccess) return e;
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_score<kFmt, true>, kScoreThreads,
                                                           smem)) != cudaSuccess)
        return e;
    const int blocks = sms * (per_sm > 0 ? per_sm : 1);
    return launch_pdl(k_score<kFmt, true>, dim3(static_cast<unsigned>(blocks)), dim3(kScoreThreads), smem,
                      stream, static_cast<const uint16_t *>(q), static_cast<const uint8_t *>(summ),
                      page_table, seq_lens, batch, hq, hkv, max_pages, weights_ld(max_pages),
                      num_pages, scale_log2, weights, chunks, chunks_ld(max_pages), kStagesMax,
                      early ? 1 : 0, status);
}

cudaError_t launch_score(const void *q, const void *summ, int fmt, const int32_t *page_table,
                         const int32_t *seq_lens, int batch, int hq, int hkv, int max_pages,
                         long long num_pages, float scale_log2, float *weights, float *chunks,
                         bool early, uint32_t *status, cudaStream_t stream)
{
    auto launch = fmt == kSummQ8 ? launch_score_fmt<kSummQ8>
                                 : (fmt == kSummQ2 ? launch_score_fmt<kSummQ2> : launch_score_fmt<kSummBf16>);
    return launch(q, summ, page_table, seq_lens, batch, hq, hkv, max_pages, num_pages, scale_log2,
                  weights, chunks, early, status, stream);
}

cudaError_t launch_select(const float *weights, const float *chunks, const int32_t *page_table,
                          const int32_t *seq_lens, int batch, int hq, int hkv, int max_pages,
                          long long num_pages, int rule, unsigned long long target, float delta,
                          bool dense, int32_t *lists, int32_t *lengths, uint32_t *status,
                          cudaStream_t stream)
{
    const int ldc = chunks_ld(max_pages);
    const size_t smem = dense ? 0 : select_smem_bytes(max_pages, ldc);
    const bool wide = max_pages > 8 * kSelThreads;            // 16 stripes of 1024 pages
    auto kernel = wide ? k_select<16> : k_select<8>;
    if (!dense) {
        static std::atomic<int> seen8[64], seen16[64];
        cudaError_t e = raise_smem_limit(kernel, smem, wide ? seen16 : seen8);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kernel, dim3(batch * hkv), dim3(kSelThreads), smem, stream, weights, chunks,
                      page_table, seq_lens, hq, hkv, max_pages, weights_ld(max_pages), ldc,
                      num_pages, rule, target, delta, dense ? 1 : 0, lists, lengths, status);
}

}  // namespace moira
