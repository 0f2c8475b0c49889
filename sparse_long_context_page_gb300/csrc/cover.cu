// The gamma-coverage selection of one layer in a single launch: one
// thread-block cluster per (request, KV head) list.
//
// "MOIRA: Mass-Oriented Indexing with Ragged Attention for Long-Context
// Decoding", abstract: per request, layer and KV head, keep the fewest pages
// whose estimated share of the attention reaches gamma.  k_score + k_select
// compute this in two launches, and for a batch of one request the second
// runs on 8 SMs (one block per list), a chain of block-wide phases that
// waits on L2 round trips.  k_cover spreads each list over the C blocks of a
// cluster (C = 16 or 8): every block scores its share of the list's 32-page
// chunks, and the blocks exchange what the cut needs through distributed
// shared memory, ordered by the cluster's hardware barrier:
//   1. scores: the block's chunks' summaries arrive by bulk copies, the G
//      query rows' logits come from mma.sync (exactly as k_score forms them),
//      then per chunk and head the max M_c, the sum Z_c and the weights
//      e_hp = 2^(s_hp - M_c) (weights stay in registers);
//   2. every block sends its chunk statistics to every block    [barrier 1]
//   3. every block merges the normalisers in k_select's fixed order, forms
//      its pages' masses and its level-1 histogram              [barrier 2]
//   4. block c sums slice c of the C histograms and sends its total to all
//                                                               [barrier 3]
//   5. every block finds the crossing slice from the totals, reads that
//      slice's summed bins from its owner, finds the crossing bin, and sends
//      its pages in that bin to every block                     [barrier 4]
//   6. every block refines the cut from the candidates (k_select's integer
//      sums, so the cut is k_select's), counts its kept pages and sends the
//      counts to all                                            [barrier 5]
//   7. every block writes its kept pages at their place in the ascending
//      list; block 0 adds the partial tail page and the length.
// The masses, the level-1 bins, the refinement and the tie rule are
// k_select's, in the same arithmetic, so the lists and lengths are bit-equal
// to k_score + k_select's.
//
// It runs for the coverage rule over bf16 summaries when every list's
// cluster is resident at once (units <= the device's active clusters of size
// C) and a block's chunks fit two rounds of 16.  It is an opt-in entry point
// (moira_select_clustered), not the decode step's selection: at batch 1 on
// GB300 it takes 21 us per 128k layer against 15 us for the two launches.
// Each phase is a chain of dependent shared-memory and DSMEM operations on
// a few warps, every exchange waits for the cluster's slowest block, and the
// summaries' 16.8 MB arrive through 64 SMs in two rounds instead of
// k_score's 152.
#include <atomic>

#include "select_core.cuh"

namespace moira {

constexpr int kCovThreads = 1024;
constexpr int kCovWarps = kCovThreads / 32;
constexpr int kCovSlots = 16;                                // chunks per round, 2 warps each
constexpr int kCovMaxRounds = 2;
constexpr int kCovMaxOwnChunks = kCovSlots * kCovMaxRounds;  // 32
constexpr int kCovMaxOwnPages = kCovMaxOwnChunks * kScoreChunk;   // 1024: one page per thread
constexpr int kCovMaxChunks = kMaxPagesPerSeq / kScoreChunk;      // 512
constexpr int kCovRow = kHeadDim * 2 + 16;                   // smem bytes per summary row (ldmatrix banks)
constexpr int kCovMaxCluster = 16;
constexpr int kCovMaxSlice = (kL1Bins + 7) / 8;              // 529 level-1 bins per block (C = 8)
static_assert(kCovMaxOwnPages == kCovThreads, "compaction: one own page per thread");
static_assert(kCovSlots * 2 == kCovWarps, "two warps (16-page halves) per chunk slot");
static_assert(kCovMaxChunks <= 2 * 256, "normalisers: two chunks per thread and head");

struct CoverShared {
    float2 cs[kGroup][kCovMaxChunks];           // every chunk's (M_c, Z_c) per head
    float4 f[kCovMaxOwnChunks];                 // own chunks' factors 2^(M_c - M_h) / (G Z_h)
    float s_s[kCovSlots][kGroup][kScoreChunk];  // a round's logits
    uint32_t bits[kCovMaxOwnPages];             // own pages' mass bit patterns
    int32_t phys[kCovMaxOwnPages];              // own pages' physical ids
    uint32_t h1[kL1Bins];
    uint32_t red[kCovMaxSlice];                 // this block's slice of the summed level-1 bins
    uint32_t cand[kCand];
    uint32_t cand_fx[kPairMax];
    uint16_t cand_idx[kCand];
    uint32_t h2[kL2Bins];
    unsigned long long tot[kCovMaxCluster];     // every block's slice total
    uint32_t cnt[kCovMaxCluster];               // every block's kept counts: gt | eq << 16
    uint32_t wcnt[kCovWarps];                   // this block's per-warp counts, then their prefix
    unsigned long long scan[kCovWarps];
    unsigned long long bar[kCovWarps];          // one mbarrier per 16-page half
    float red_m[kCovWarps];
    float red_z[kCovWarps];
    unsigned long long above;
    uint32_t lo, hi;
    int found;
    int ncand;
    int abort;
};

constexpr size_t kCovStageBytes = static_cast<size_t>(kCovSlots) * kScoreChunk * kCovRow;
constexpr size_t kCovSmemBytes = kCovStageBytes + sizeof(CoverShared);

// ---- distributed shared memory ---------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_blocks()
{
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}
// The shared::cluster address of `local`'s counterpart in block `rank`.
__device__ __forceinline__ uint32_t dsm(const void *local, uint32_t rank)
{
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
    return a;
}
__device__ __forceinline__ void dsm_st(uint32_t a, uint32_t v)
{
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void dsm_st(uint32_t a, uint16_t v)
{
    asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}
__device__ __forceinline__ void dsm_st(uint32_t a, unsigned long long v)
{
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}
__device__ __forceinline__ void dsm_st(uint32_t a, float2 v)
{
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(a), "f"(v.x), "f"(v.y) : "memory");
}
__device__ __forceinline__ uint32_t dsm_ld(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t dsm_atomic_add(uint32_t a, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(a), "r"(v) : "memory");
    return old;
}
// Cluster barrier: the release half orders this thread's earlier writes
// (local and remote) before the acquire half of every thread's wait.  Every
// thread of every block of the cluster takes part, each the same number of
// times (the forms without .aligned: a warp need not be converged).
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Exclusive scan over the block (1024 threads) in thread order; *total gets
// the sum.
__device__ __forceinline__ unsigned long long cov_excl_scan(unsigned long long v, unsigned long long *s_warp,
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
    *total = s_warp[kCovWarps - 1];
    __syncthreads();
    return off + x - v;
}

template <int kRounds>
__global__ void __launch_bounds__(kCovThreads, 1) k_cover(
    const uint16_t *__restrict__ q, const uint8_t *__restrict__ summ, const int32_t *__restrict__ page_table,
    const int32_t *__restrict__ seq_lens, int hq, int hkv, int max_pages, long long num_pages, float scale_log2,
    unsigned long long target, int early, int32_t *__restrict__ lists, int32_t *__restrict__ lengths,
    uint32_t *status)
{
    extern __shared__ __align__(128) uint8_t s_cov[];
    uint8_t *stage = s_cov;                                                // [16 slots][32 pages][kCovRow]
    CoverShared &sh = *reinterpret_cast<CoverShared *>(s_cov + kCovStageBytes);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t C = cluster_blocks(), rank = cluster_rank();
    const int u = static_cast<int>(blockIdx.x / C);
    const int r = u / hkv, j = u % hkv;
    const int32_t *row = page_table + static_cast<size_t>(r) * max_pages;
    int32_t *out = lists + static_cast<size_t>(u) * max_pages;
    const WaitGuard wg{&sh.abort, status};

    if (!early) pdl_wait();
    int L = __ldg(seq_lens + r);
    if (L < 0 || L > max_pages * kPageSize) {
        if (tid == 0 && rank == 0) raise_status(status, kDevBadLen);
        L = L < 0 ? 0 : max_pages * kPageSize;
    }
    const int F = L / kPageSize, T = (L % kPageSize) != 0;
    if (F == 0) {                                       // cluster-uniform: only the tail page
        if (early) pdl_wait();
        pdl_trigger();
        if (rank == 0 && tid == 0) {
            if (T) out[0] = __ldg(row);
            lengths[u] = T;
        }
        return;
    }
    const int nch = (F + kScoreChunk - 1) / kScoreChunk;
    const int ch0 = static_cast<int>(rank * nch / C), ch1 = static_cast<int>((rank + 1) * nch / C);
    const int own = (ch1 - ch0) * kScoreChunk;          // own page slots (the last chunk may be partial)

    if (tid == 0) guard_init(wg);
    if (lane == 0) mbar_init(smem_u32(&sh.bar[warp]), 1);
    for (int b = tid; b < kL1Bins; b += kCovThreads) sh.h1[b] = 0u;
    if (tid == 0) sh.ncand = 0;
    mbar_fence_init();
    __syncthreads();
    cluster_arrive_relaxed();                           // every block has started: remote writes may follow

    // ---- 1. scores of the own chunks, in rounds of 16 ---------------------------------
    const int slot = warp >> 1, half = warp & 1;
    const int hrow = (lane >> 2) & 3, t4 = lane & 3;
    uint32_t qw[16];
    float ew[kRounds][4];                               // stats warps: weights of (head lane/8, pages 4*(lane%8)..)
    const uint32_t bar = smem_u32(&sh.bar[warp]);
    int32_t pid[kRounds];
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
        const int cg = ch0 + rd * kCovSlots + slot;
        const int p = cg * kScoreChunk + half * 16 + (lane & 15);
        pid[rd] = (cg < ch1 && lane < 16 && p < F) ? __ldg(row + p) : -1;
    }
    if (early) pdl_wait();
    pdl_trigger();
    {
        const uint16_t *qa = q + (static_cast<size_t>(r) * hq + j * kGroup + hrow) * kHeadDim + 2 * t4;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qw[2 * ks] = __ldg(reinterpret_cast<const uint32_t *>(qa + ks * 16));
            qw[2 * ks + 1] = __ldg(reinterpret_cast<const uint32_t *>(qa + ks * 16 + 8));
        }
    }
    const size_t rec = static_cast<size_t>(hkv) * kHeadDim * 2;
#pragma unroll
    for (int rd = 0; rd < kRounds; ++rd) {
        const int cg = ch0 + rd * kCovSlots + slot;
        const bool has = cg < ch1;                      // warp-uniform
        uint32_t okm = 0u;
        if (has) {
            const int p = cg * kScoreChunk + half * 16 + (lane & 15);
            const bool in = lane < 16 && p < F;
            const bool ok = in && pid[rd] >= 0 && pid[rd] < num_pages;
            if (in && !ok) raise_status(status, kDevBadPage);
            okm = __ballot_sync(0xffffffffu, ok);
            if (lane < 16) sh.phys[(rd * kCovSlots + slot) * kScoreChunk + half * 16 + lane] = pid[rd];
            if (lane == 0) mbar_arrive_expect_tx(bar, __popc(okm) * kHeadDim * 2);
            __syncwarp();
            if (ok)
                bulk_load(smem_u32(stage + (slot * kScoreChunk + half * 16 + lane) * kCovRow),
                          summ + static_cast<size_t>(pid[rd]) * rec + static_cast<size_t>(j) * kHeadDim * 2,
                          kHeadDim * 2, bar);
            mbar_wait_g(bar, static_cast<uint32_t>(rd) & 1u, wg);
            float acc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
            const int prow = half * 16 + (lane & 7) + ((lane >> 4) << 3);
            const uint32_t rbase = smem_u32(stage) + (slot * kScoreChunk + prow) * kCovRow + (((lane >> 3) & 1) << 4);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(rbase + ks * 32, b0, b1, b2, b3);
                mma_bf16_16816(acc[0], qw[2 * ks], 0u, qw[2 * ks + 1], 0u, b0, b1);
                mma_bf16_16816(acc[1], qw[2 * ks], 0u, qw[2 * ks + 1], 0u, b2, b3);
            }
            if (lane < 16) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int pl = nt * 8 + 2 * t4;             // within the half
                    float s0 = acc[nt][0] * scale_log2, s1 = acc[nt][1] * scale_log2;
                    if (!((okm >> pl) & 1u)) s0 = -INFINITY;
                    if (!((okm >> (pl + 1)) & 1u)) s1 = -INFINITY;
                    *reinterpret_cast<float2 *>(&sh.s_s[slot][hrow][half * 16 + pl]) = make_float2(s0, s1);
                }
            }
        }
        __syncthreads();                                // logits complete; the stage may be refilled
        // chunk statistics of slot `warp` (warps 0..15): 8 lanes per head, 4 pages per lane
        if (warp < kCovSlots) {
            const int cgs = ch0 + rd * kCovSlots + warp;
            const int hl = lane >> 3, sub = lane & 7;
            ew[rd][0] = ew[rd][1] = ew[rd][2] = ew[rd][3] = 0.f;
            if (cgs < ch1) {                            // warp-uniform
                const float4 v = *reinterpret_cast<const float4 *>(&sh.s_s[warp][hl][sub * 4]);
                float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                const float ms = mx == -INFINITY ? 0.f : mx;
                ew[rd][0] = exp2f(v.x - ms);
                ew[rd][1] = exp2f(v.y - ms);
                ew[rd][2] = exp2f(v.z - ms);
                ew[rd][3] = exp2f(v.w - ms);
                float sum = (ew[rd][0] + ew[rd][1]) + (ew[rd][2] + ew[rd][3]);
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                if (sub == 0) sh.cs[hl][cgs] = make_float2(mx, sum);
            }
        }
        __syncthreads();                                // s_s read before the next round writes it
    }

    // ---- 2. every block gets every chunk's statistics ---------------------------------
    cluster_wait();                                     // all blocks have started
    {
        const int n = (ch1 - ch0) * kGroup * static_cast<int>(C);
        for (int i = tid; i < n; i += kCovThreads) {
            const uint32_t dst = static_cast<uint32_t>(i) % C;
            const int rest = i / static_cast<int>(C), h = rest % kGroup, c = ch0 + rest / kGroup;
            if (dst != rank) dsm_st(dsm(&sh.cs[h][c], dst), sh.cs[h][c]);
        }
    }
    cluster_sync();                                     // [barrier 1]

    // ---- 3. normalisers (k_select's fixed order), masses, level-1 histogram ----------
    {
        const int hg = tid >> 8, ci = tid & 255;
        float cm[2] = {-INFINITY, -INFINITY}, cz[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = ci + 256 * i;
            if (c < nch) {
                const float2 v = sh.cs[hg][c];
                cm[i] = v.x;
                cz[i] = v.y;
            }
        }
        const float mx = warp_max_butterfly(fmaxf(cm[0], cm[1]));
        if (lane == 0) sh.red_m[warp] = mx;
        __syncthreads();
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 8; ++w) M = fmaxf(M, sh.red_m[hg * 8 + w]);
        const float z = warp_sum_butterfly(chunk_weight_sum(cm[0], cz[0], cm[1], cz[1], M));
        if (lane == 0) sh.red_z[warp] = z;
        __syncthreads();
        const float zinv = head_zinv(&sh.red_z[hg * 8]);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int c = ci + 256 * i;
            if (c >= ch0 && c < ch1) reinterpret_cast<float *>(sh.f)[4 * (c - ch0) + hg] = chunk_factor(cm[i], M, zinv);
        }
    }
    __syncthreads();
    if (warp < kCovSlots) {
        const int sub = lane & 7;
#pragma unroll
        for (int rd = 0; rd < kRounds; ++rd) {
            const int cg = ch0 + rd * kCovSlots + warp;
            if (cg >= ch1) break;                       // warp-uniform
            const float4 f = sh.f[cg - ch0];
            float w1[4], w2[4], w3[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                w1[i] = __shfl_sync(0xffffffffu, ew[rd][i], sub + 8);
                w2[i] = __shfl_sync(0xffffffffu, ew[rd][i], sub + 16);
                w3[i] = __shfl_sync(0xffffffffu, ew[rd][i], sub + 24);
            }
            const int p = cg * kScoreChunk + sub * 4;
            uint32_t xs[4] = {0u, 0u, 0u, 0u};
            if (lane < 8) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    xs[i] = p + i < F ? page_mass_bits(ew[rd][i], w1[i], w2[i], w3[i], f) : 0u;
                *reinterpret_cast<uint4 *>(&sh.bits[(cg - ch0) * kScoreChunk + sub * 4]) =
                    make_uint4(xs[0], xs[1], xs[2], xs[3]);
            }
            // masses below 2^-32 are 0 in fixed point and add nothing
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t fx = to_fx(xs[i]);
                hist_add_warp(sh.h1, static_cast<uint32_t>(l1_bin(xs[i])), fx, lane < 8 && p + i < F && fx != 0u);
            }
        }
    }
    __syncthreads();
    cluster_sync();                                     // [barrier 2] every level-1 histogram is complete

    // ---- 4. block `rank` sums its slice of the bins over the cluster -----------------
    const int SL = (kL1Bins + static_cast<int>(C) - 1) / static_cast<int>(C);
    {
        const int b0 = static_cast<int>(rank) * SL, nb = min(kL1Bins - b0, SL);
        uint32_t v = 0u;
        if (tid < nb) {
            for (uint32_t rk = 0; rk < C; ++rk) v += dsm_ld(dsm(&sh.h1[b0 + tid], rk));
            sh.red[tid] = v;
        }
        unsigned long long total;
        cov_excl_scan(v, sh.scan, &total);
        if (tid < static_cast<int>(C)) dsm_st(dsm(&sh.tot[rank], static_cast<uint32_t>(tid)), total);
    }
    cluster_sync();                                     // [barrier 3]

    // ---- 5. the crossing bin, then its pages to every block -------------------------
    int cstar = -1;
    unsigned long long above0 = 0ull;
    {
        unsigned long long acc = 0ull;
        for (int c = static_cast<int>(C) - 1; c >= 0; --c) {       // slices from the top
            const unsigned long long tv = sh.tot[c];
            if (acc < target && acc + tv >= target) {
                cstar = c;
                above0 = acc;
                break;
            }
            acc += tv;
        }
    }
    if (tid == 0) sh.found = cstar >= 0;
    if (cstar >= 0) {                                   // block-uniform
        const int b0 = cstar * SL, nb = min(kL1Bins - b0, SL);
        const uint32_t v = tid < nb ? dsm_ld(dsm(&sh.red[nb - 1 - tid], static_cast<uint32_t>(cstar))) : 0u;
        unsigned long long total;
        const unsigned long long acc = above0 + cov_excl_scan(v, sh.scan, &total);
        if (tid < nb && acc < target && acc + v >= target) {
            const int b = b0 + nb - 1 - tid;
            sh.lo = l1_lo(b);
            sh.hi = l1_hi(b);
            sh.above = acc;
        }
        __syncthreads();
        const uint32_t lo = sh.lo, hi = sh.hi;
        const int p = ch0 * kScoreChunk + tid;
        const uint32_t x = tid < own && p < F ? sh.bits[tid] : 0u;
        const bool in = tid < own && p < F && x >= lo && x < hi;
        const unsigned m = __ballot_sync(0xffffffffu, in);
        if (m) {                                        // warp-uniform
            uint32_t base = 0u;
            if (lane == 0) base = dsm_atomic_add(dsm(&sh.ncand, 0u), static_cast<uint32_t>(__popc(m)));
            base = __shfl_sync(0xffffffffu, base, 0);
            const uint32_t slot_c = base + static_cast<uint32_t>(__popc(m & ((1u << lane) - 1u)));
            if (in && slot_c < static_cast<uint32_t>(kCand)) {
                const uint32_t fx = to_fx(x);
                for (uint32_t rk = 0; rk < C; ++rk) {
                    dsm_st(dsm(&sh.cand[slot_c], rk), x);
                    dsm_st(dsm(&sh.cand_idx[slot_c], rk), static_cast<uint16_t>(p));
                    if (slot_c < static_cast<uint32_t>(kPairMax)) dsm_st(dsm(&sh.cand_fx[slot_c], rk), fx);
                }
            }
        }
    }
    cluster_sync();                                     // [barrier 4] candidates everywhere

    // ---- 6. the cut, identical in every block ----------------------------------------
    if (sh.found) {                                     // block-uniform
        const int nc = static_cast<int>(dsm_ld(dsm(&sh.ncand, 0u)));
        if (nc <= kPairMax) {
            // candidate c: masses ranked before it (larger, or equal with a lower
            // page index); the one whose running sum crosses gamma is the cut
            const unsigned long long a0 = sh.above;
            __syncthreads();
            const int lg = nc <= 32 ? 5 : nc <= 64 ? 4 : nc <= 128 ? 3 : 2;
            const int ci = tid >> lg, part = tid & ((1 << lg) - 1);
            uint32_t gt_sum = 0u, tie_before = 0u;
            uint32_t x = 0u, xi = 0u;
            if (ci < nc) {
                x = sh.cand[ci];
                xi = sh.cand_idx[ci];
                for (int c = part; c < nc; c += 1 << lg) {
                    const uint32_t y = sh.cand[c], fy = sh.cand_fx[c];
                    gt_sum += y > x ? fy : 0u;
                    tie_before += (y == x && sh.cand_idx[c] < xi) ? fy : 0u;
                }
            }
            for (int o = 1; o < (1 << lg); o <<= 1) {
                gt_sum += __shfl_xor_sync(0xffffffffu, gt_sum, o);
                tie_before += __shfl_xor_sync(0xffffffffu, tie_before, o);
            }
            if (ci < nc && part == 0) {
                const unsigned long long before = a0 + gt_sum + tie_before;
                if (before < target && before + sh.cand_fx[ci] >= target) {
                    sh.lo = x;
                    sh.hi = x + 1u;
                    sh.above = a0 + gt_sum;
                }
            }
            __syncthreads();
        } else if (nc <= kCand) {
            if (warp == 0) {
                uint32_t lo = sh.lo, hi = sh.hi;
                unsigned long long above = sh.above;
                warp_refine(sh.cand, nc, sh.h2, kRuleCoverage, target, lo, hi, above);
                if (lane == 0) {
                    sh.lo = lo;
                    sh.hi = hi;
                    sh.above = above;
                    if (hi - lo > 1u && rank == 0) raise_status(status, kDevBadLen);
                }
            }
            __syncthreads();
        } else {
            // more tied pages than candidates: 256-bin passes over every block's masses
            for (int pass = 0; sh.hi - sh.lo > 1u; ++pass) {
                if (pass >= 6) {                        // cannot happen: exact integer sums
                    if (tid == 0 && rank == 0) raise_status(status, kDevBadLen);
                    break;
                }
                const uint32_t lo = sh.lo, hi = sh.hi;
                int shift, nb;
                refine_bins(lo, hi, shift, nb);
                if (tid < kL2Bins) sh.h2[tid] = 0u;
                __syncthreads();
                for (uint32_t rk = 0; rk < C; ++rk) {
                    const int k0 = static_cast<int>(rk * nch / C), k1 = static_cast<int>((rk + 1) * nch / C);
                    const int p = k0 * kScoreChunk + tid;
                    const bool mine = tid < (k1 - k0) * kScoreChunk && p < F;
                    const uint32_t x = mine ? dsm_ld(dsm(&sh.bits[tid], rk)) : 0u;
                    hist_add_warp(sh.h2, (x - lo) >> shift, to_fx(x), mine && x >= lo && x < hi);
                }
                __syncthreads();
                if (warp == 0) {
                    uint32_t l2 = lo, h2 = hi;
                    unsigned long long above = sh.above;
                    warp_pick_bin([&](int b) { return sh.h2[b]; }, nb, shift, target, l2, h2, above);
                    if (lane == 0) {
                        sh.lo = l2;
                        sh.hi = h2;
                        sh.above = above;
                    }
                }
                __syncthreads();
            }
        }
    }
    uint32_t cut, need_tied;
    if (sh.found) {
        cut = sh.lo;
        const uint32_t cfx = to_fx(cut);                // > 0: it carried the crossing
        const uint32_t d = static_cast<uint32_t>(target - sh.above);
        need_tied = d / cfx + (d % cfx != 0u ? 1u : 0u);
    } else {                                            // total < gamma: keep all
        cut = 0u;
        need_tied = 0xFFFFFFFFu;
    }

    // ---- 7. kept counts to every block, then the ordered writes -----------------------
    const int p = ch0 * kScoreChunk + tid;
    const bool valid = tid < own && p < F;
    const uint32_t x = valid ? sh.bits[tid] : 0u;
    const unsigned gt_m = __ballot_sync(0xffffffffu, valid && x > cut);
    const unsigned eq_m = __ballot_sync(0xffffffffu, valid && x == cut);
    if (lane == 0) sh.wcnt[warp] = static_cast<uint32_t>(__popc(gt_m)) | (static_cast<uint32_t>(__popc(eq_m)) << 16);
    __syncthreads();
    if (warp == 0) {
        const uint32_t c = sh.wcnt[lane];
        uint32_t xs = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, xs, o);
            if (lane >= o) xs += y;
        }
        sh.wcnt[lane] = xs - c;
        const uint32_t total = __shfl_sync(0xffffffffu, xs, 31);
        if (lane < static_cast<int>(C)) dsm_st(dsm(&sh.cnt[rank], static_cast<uint32_t>(lane)), total);
    }
    cluster_sync();                                     // [barrier 5] no shared memory is read remotely after it
    uint32_t gt_base = 0u, eq_base = 0u, gt_all = 0u, eq_all = 0u;
    for (uint32_t c = 0; c < C; ++c) {
        const uint32_t v = sh.cnt[c];
        if (c < rank) {
            gt_base += v & 0xFFFFu;
            eq_base += v >> 16;
        }
        gt_all += v & 0xFFFFu;
        eq_all += v >> 16;
    }
    if ((gt_m | eq_m) != 0u) {                          // warp-uniform
        const unsigned lt = (1u << lane) - 1u;
        const uint32_t base = sh.wcnt[warp];
        const uint32_t gt_before = gt_base + (base & 0xFFFFu) + __popc(gt_m & lt);
        const uint32_t eq_before = eq_base + (base >> 16) + __popc(eq_m & lt);
        const bool is_gt = (gt_m >> lane) & 1u, is_eq = (eq_m >> lane) & 1u;
        if (is_gt || (is_eq && eq_before < need_tied)) {
            const int32_t pg = sh.phys[tid];
            if (pg < 0 || pg >= num_pages) raise_status(status, kDevBadPage);
            out[gt_before + (eq_before < need_tied ? eq_before : need_tied)] = pg;
        }
    }
    if (rank == 0 && tid == 0) {
        const int kept = static_cast<int>(gt_all + (eq_all < need_tied ? eq_all : need_tied));
        if (T) out[kept] = __ldg(row + F);
        lengths[u] = kept + T;
    }
    // after a give-up, let this warp's copies still in flight land before the block exits
    if (lane == 0 && guard_failed(wg)) {
        const uint64_t deadline = globaltimer() + kDrainLimitNs;
        int last = -1;
        for (int rd = 0; rd < kRounds; ++rd)
            if (ch0 + rd * kCovSlots + slot < ch1) last = rd;
        if (last >= 0) mbar_drain(bar, static_cast<uint32_t>(last) & 1u, deadline);
    }
}

// ---------------------------------------------------------------------------
// Host side: which cluster size a launch takes, and the launch.
// ---------------------------------------------------------------------------
namespace {
// Per device, cluster size (index 0: 16, 1: 8) and kernel instance (rounds
// 1 or 2, each with its own attributes): 0 unknown, -1 unusable, else 1 +
// the number of clusters that fit at once.  Internal linkage: no other
// library in the process shares it.
std::atomic<int> g_cover_fit[64][2][kCovMaxRounds];

template <int kRounds>
int cover_active_clusters(int dev, int c_idx)
{
    std::atomic<int> &slot = g_cover_fit[dev][c_idx][kRounds - 1];
    const int seen = slot.load(std::memory_order_relaxed);
    if (seen != 0) return seen - 1;
    const int C = c_idx == 0 ? 16 : 8;
    int fit = -1;
    auto kern = k_cover<kRounds>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kCovSmemBytes)) == cudaSuccess &&
        (C <= 8 || cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess)) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C);
        cfg.blockDim = dim3(kCovThreads);
        cfg.dynamicSmemBytes = kCovSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess) fit = n;
    }
    (void)cudaGetLastError();                           // a refused attribute is not an error of the caller
    slot.store(fit + 1, std::memory_order_relaxed);
    return fit;
}

int cover_rounds(int max_pages, int C)
{
    const int nch = (max_pages + kScoreChunk - 1) / kScoreChunk;
    const int own = (nch + C - 1) / C;
    return (own + kCovSlots - 1) / kCovSlots;
}
}  // namespace

int cover_cluster_size(int units, int max_pages)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int sizes[2] = {16, 8};
    for (int c_idx = 0; c_idx < 2; ++c_idx) {
        const int C = sizes[c_idx];
        const int rounds = cover_rounds(max_pages, C);
        if (rounds > kCovMaxRounds) continue;
        const int fit = rounds == 1 ? cover_active_clusters<1>(dev, c_idx) : cover_active_clusters<2>(dev, c_idx);
        if (fit >= units) return C;
    }
    return 0;
}

cudaError_t launch_cover(const void *q, const void *summ, const int32_t *page_table, const int32_t *seq_lens,
                         int batch, int hq, int hkv, int max_pages, long long num_pages, float scale_log2,
                         unsigned long long target, bool early, int32_t *lists, int32_t *lengths,
                         uint32_t *status, int C, cudaStream_t stream)
{
    const int units = batch * hkv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units * C));
    cfg.blockDim = dim3(kCovThreads);
    cfg.dynamicSmemBytes = kCovSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const uint16_t *qq = static_cast<const uint16_t *>(q);
    const uint8_t *ss = static_cast<const uint8_t *>(summ);
    if (cover_rounds(max_pages, C) == 1)
        return cudaLaunchKernelEx(&cfg, k_cover<1>, qq, ss, page_table, seq_lens, hq, hkv, max_pages, num_pages,
                                  scale_log2, target, early ? 1 : 0, lists, lengths, status);
    return cudaLaunchKernelEx(&cfg, k_cover<2>, qq, ss, page_table, seq_lens, hq, hkv, max_pages, num_pages,
                              scale_log2, target, early ? 1 : 0, lists, lengths, status);
}

}  // namespace moira
