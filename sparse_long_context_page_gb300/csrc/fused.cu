// The selection and the attention of one layer in one launch, for small
// batches ("MOIRA: Mass-Oriented Indexing with Ragged Attention for
// Long-Context Decoding", abstract: a coverage rule keeps the fewest pages
// whose estimated attention mass reaches gamma, and a self-planning ragged
// attention kernel reads only those pages, the whole step staying inside one
// CUDA graph; the abstract also names the cost this fusion attacks: adaptive
// budgets pay with extra selection cost).
//
// With one request, k_select runs one block per (request, KV head) on 8 SMs
// while the rest of the GPU and HBM wait, and the attention launch that
// follows pays its own start.  Here the grid of the attention kernel (2 blocks
// per SM, all resident together) does both, after k_score has written the
// chunk statistics and the chunk-relative weights:
//
//  1. list u gets cpu = grid / units blocks, block c taking an equal run of
//     u's 32-page chunks.  Every block reduces u's chunk statistics to the
//     head normalisers in the fixed order k_select uses, forms the masses of
//     its own pages exactly as k_select does, writes them to u's mass row and
//     adds their fixed-point values into u's level-1 histogram (global
//     memory).                                            barrier (list u)
//  2. every block copies u's whole mass row and histogram into shared memory
//     and finds the cut itself, as k_select does: the crossing bin of the
//     histogram, then the exact bit pattern among the bin's pages.  The cut
//     is reached through exact integer sums, so every block of the list gets
//     the same one and the lists are bit-identical to moira_select's.
//  3. every block writes its run's kept pages at their places in the
//     ascending list (it can count the kept pages before its run), the first
//     block the length, the last the partial tail page.    barrier (grid)
//  4. the attention of k_attend over those lists (same plan, same order, so
//     the output equals moira_select + moira_attend bit for bit).
// Every wait is bounded (WaitGuard): a barrier that never completes records
// MOIRA_DEV_TIMEOUT and the launch ends with its results marked invalid.
#include "attend_core.cuh"
#include "select_core.cuh"

namespace moira {

constexpr int kFusedSlots = kFewSlots, kFusedWarps = kFewWarps;
constexpr int kFusedThreads = (kFusedWarps + 1) * 32;            // 160
constexpr int kFusedAllWarps = kFusedWarps + 1;
constexpr int kFusedChunks = 16;                                  // chunks per selecting block, at most
constexpr int kFusedPages = kFusedChunks * kScoreChunk;           // 512: 4 per consumer thread
constexpr int kFusedMaxBlocks = 384;
constexpr int kFusedUnitPer = (kFusedMaxUnits + 31) / 32;
constexpr int kL1Per = (kL1Bins + kFusedThreads - 1) / kFusedThreads;   // 27 level-1 bins per thread
static_assert(kFusedPages == 4 * kFusedWarps * 32, "one group of 4 pages per consumer thread");
static_assert(kFusedMaxUnits < kManyUnits, "the fused kernel runs the few-list block shape");

// Scratch of the selection inside the stage ring (idle until the attention):
// the list's masses, its level-1 histogram, the crossing bin's candidates.
constexpr int kRingMass = 0;                                      // uint32 [kMaxPagesPerSeq]
constexpr int kRingH1 = kRingMass + kMaxPagesPerSeq * 4;          // uint32 [kL1Stride]
constexpr int kRingCand = kRingH1 + kL1Stride * 4;                // uint32 [kCand]
constexpr int kRingH2 = kRingCand + kCand * 4;                    // uint32 [kL2Bins]
constexpr int kRingCm = kRingH2 + kL2Bins * 4;                    // float [4][kFusedChunks]
constexpr int kRingF = kRingCm + kGroup * kFusedChunks * 4;       // float4 [kFusedChunks]
static_assert(kRingF + kFusedChunks * 16 <= kFusedSlots * kSlotBytes, "selection scratch fits the ring");
static_assert(kRingH1 % 16 == 0 && (kL1Stride * 4) % 16 == 0, "bulk copies of whole 16-byte units");

struct FusedShared {
    unsigned long long above;
    unsigned long long scan64[kFusedAllWarps];
    uint32_t scan32[kFusedAllWarps];
    uint32_t lo, hi, cut, need;
    int found, ncand;
    float red[32], red2[32], M[kGroup], zinv[kGroup];
    unsigned long long load_bar;        // the bulk copy of a list's masses and histogram
};

// Exclusive scan over the block (all warps) in thread order.
template <typename T>
__device__ __forceinline__ T fused_excl_scan(T v, T *s_w, T &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    T off = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kFusedAllWarps; ++w) {
        if (w < warp) off += s_w[w];
        tot += s_w[w];
    }
    __syncthreads();
    total = tot;
    return off + x - v;
}

// Exclusive warp scan of per-lane values; `total` gets the warp's sum.
__device__ __forceinline__ int warp_excl_scan(int v, int &total)
{
    const int lane = threadIdx.x & 31;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    total = __shfl_sync(0xffffffffu, x, 31);
    return x - v;
}

// First chunk of block c's run when nch chunks are split over cpu blocks.
__device__ __forceinline__ int run_chunk(int c, int nch, int cpu) { return c * nch / cpu; }

// Full pages and partial-tail tokens of a request of L tokens (clamped).
__device__ __forceinline__ void request_pages(int L, int mp, int &F, int &tail)
{
    L = L < 0 ? 0 : (L > mp * kPageSize ? mp * kPageSize : L);
    F = L / kPageSize;
    tail = L % kPageSize;
}

template <int kSlots, int kConsumerWarps>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, kBlocksPerSm)
    k_select_attend(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                    const FusedArgs f)
{
    static_assert(kSlots == kFusedSlots && kConsumerWarps == kFusedWarps, "one block shape");
    constexpr int kThreads = kFusedThreads;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *stage = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    AttendSmem<kSlots, kConsumerWarps> &sm =
        *reinterpret_cast<AttendSmem<kSlots, kConsumerWarps> *>(stage + kSlots * kSlotBytes);
    const AttendArgs &a = f.at;
    const int U = a.units;
    const int nblk = gridDim.x;
    const int cpu = nblk / U;                      // blocks per list in the selection
    const int n_sel = f.dense ? 0 : U * cpu;
    int *s_off = reinterpret_cast<int *>(&sm + 1);                 // [U + 1] list offsets
    int *s_utail = s_off + U + 1;                                  // [U] tokens of the partial tail page
    uint32_t *s_mass = reinterpret_cast<uint32_t *>(stage + kRingMass);
    uint32_t *s_h1 = reinterpret_cast<uint32_t *>(stage + kRingH1);
    uint32_t *s_cand = reinterpret_cast<uint32_t *>(stage + kRingCand);
    uint32_t *s_h2 = reinterpret_cast<uint32_t *>(stage + kRingH2);
    float *s_cm = reinterpret_cast<float *>(stage + kRingCm);
    float4 *s_f = reinterpret_cast<float4 *>(stage + kRingF);
    __shared__ FusedShared sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x;
    const int mp = a.max_pages;
    const WaitGuard wg{&sm.abort, a.status};
    uint32_t *grid_bar = f.bars + kFusedMaxUnits * kBarWords;

    attend_init(sm, &tmap_k, &tmap_v, a.status);
    if (tid == 0) {
        sh.found = 0;
        sh.ncand = 0;
        mbar_init(smem_u32(&sh.load_bar), 1);
        mbar_fence_init();
    }
    pdl_trigger();

    // ---- this block's share of the selection --------------------------------
    const bool selb = b < n_sel;                   // block-uniform
    const int u = selb ? b / cpu : 0, c = selb ? b % cpu : 0;
    const int r = u / a.hkv, j = u % a.hkv;
    uint32_t *unit_bar = f.bars + u * kBarWords;
    int F = 0, tail = 0, P0 = 0, P1 = 0, ch0 = 0, ch1 = 0;
    int32_t pref[4] = {0, 0, 0, 0};
    if (selb) {
        // k_score ran before this launch and waited for the caller's kernels
        // before it let this one start, so the page table and the lengths are
        // final here
        request_pages(__ldg(a.seq_lens + r), mp, F, tail);
        const int nch = (F + kScoreChunk - 1) / kScoreChunk;
        ch0 = run_chunk(c, nch, cpu);
        ch1 = run_chunk(c + 1, nch, cpu);
        P0 = ch0 * kScoreChunk;
        P1 = min(F, ch1 * kScoreChunk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int p = P0 + 4 * tid + i;
            if (p < P1) pref[i] = __ldg(f.page_table + static_cast<size_t>(r) * mp + p);
        }
        for (int i = tid; i < kL1Stride; i += kThreads) s_h1[i] = 0u;
    }
    pdl_wait();                                    // weights and chunk statistics come from k_score;
                                                   // a dense launch reads its inputs only after it
    // thread 0: the barriers' generations (the previous launch is complete)
    uint32_t gen_unit = 0u, gen_grid = 0u;
    if (tid == 0 && !f.dense) {
        if (selb) gen_unit = barrier_generation(unit_bar);
        gen_grid = barrier_generation(grid_bar);
    }
    const unsigned long long target = f.target;
    const int p4 = P0 + 4 * tid;                   // this thread's 4 pages of the run

    if (selb) {
        // ---- 1. normalisers, own masses, level-1 histogram ------------------
        const int hq = a.hq;
        const int nch = (F + kScoreChunk - 1) / kScoreChunk;
        const float *crow = f.chunks + (static_cast<size_t>(r) * hq + j * kGroup) * f.ldc;
        // virtual warps vw = warp + 5k (head vw / 8, group vw % 8) of the
        // fixed-order reduction: lane l holds chunks 32 (vw % 8) + l and + 256
        float2 cs[7][2];
#pragma unroll
        for (int k = 0; k < 7; ++k) {
            const int vw = warp + kFusedAllWarps * k;
            const int h = vw >> 3, ci = (vw & 7) * 32 + lane;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int cg = ci + 256 * i;
                cs[k][i] = make_float2(-INFINITY, 0.f);
                if (vw < 32 && cg < nch)
                    cs[k][i] = __ldg(reinterpret_cast<const float2 *>(crow + static_cast<size_t>(h) * f.ldc + 2 * cg));
            }
        }
        float4 w[kGroup];
#pragma unroll
        for (int h = 0; h < kGroup; ++h) {
            w[h] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (p4 < P1)
                w[h] = __ldg(reinterpret_cast<const float4 *>(
                    f.weights + (static_cast<size_t>(r) * hq + j * kGroup + h) * f.ld + p4));
        }
#pragma unroll
        for (int k = 0; k < 7; ++k) {
            const int vw = warp + kFusedAllWarps * k;
            if (vw < 32) {
                const float mx = warp_max_butterfly(fmaxf(cs[k][0].x, cs[k][1].x));
                if (lane == 0) sh.red[vw] = mx;
                const int h = vw >> 3, ci = (vw & 7) * 32 + lane;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int cg = ci + 256 * i;
                    if (cg >= ch0 && cg < ch1) s_cm[h * kFusedChunks + cg - ch0] = cs[k][i].x;
                }
            }
        }
        __syncthreads();
        if (tid < kGroup) {
            float M = -INFINITY;
#pragma unroll
            for (int w8 = 0; w8 < 8; ++w8) M = fmaxf(M, sh.red[tid * 8 + w8]);
            sh.M[tid] = M;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 7; ++k) {
            const int vw = warp + kFusedAllWarps * k;
            if (vw < 32) {
                const float z = warp_sum_butterfly(
                    chunk_weight_sum(cs[k][0].x, cs[k][0].y, cs[k][1].x, cs[k][1].y, sh.M[vw >> 3]));
                if (lane == 0) sh.red2[vw] = z;
            }
        }
        __syncthreads();
        if (tid < kGroup) sh.zinv[tid] = head_zinv(&sh.red2[tid * 8]);
        __syncthreads();
        if (tid < kGroup * kFusedChunks) {
            const int cl = tid >> 2, h = tid & 3;
            if (cl < ch1 - ch0)
                reinterpret_cast<float *>(s_f)[4 * cl + h] =
                    chunk_factor(s_cm[h * kFusedChunks + cl], sh.M[h], sh.zinv[h]);
        }
        __syncthreads();
        uint32_t xs[4] = {0u, 0u, 0u, 0u};
        if (p4 < P1) {
            const float4 fc = s_f[tid >> 3];
            xs[0] = page_mass_bits(w[0].x, w[1].x, w[2].x, w[3].x, fc);
            xs[1] = page_mass_bits(w[0].y, w[1].y, w[2].y, w[3].y, fc);
            xs[2] = page_mass_bits(w[0].z, w[1].z, w[2].z, w[3].z, fc);
            xs[3] = page_mass_bits(w[0].w, w[1].w, w[2].w, w[3].w, fc);
            *reinterpret_cast<uint4 *>(f.mass + static_cast<size_t>(u) * f.ld + p4) =
                make_uint4(xs[0], xs[1], xs[2], xs[3]);
        }
        // masses below 2^-32 are 0 in fixed point and add nothing
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t fx = to_fx(xs[i]);
            hist_add_warp(s_h1, static_cast<uint32_t>(l1_bin(xs[i])), fx, p4 + i < P1 && fx != 0u);
        }
        __syncthreads();
        uint32_t *gh1 = f.l1hist + static_cast<size_t>(u) * kL1Stride;
        for (int q = tid; q < kL1Stride / 4; q += kThreads) {
            const uint4 v = reinterpret_cast<const uint4 *>(s_h1)[q];
            if (v.x) atomicAdd(gh1 + 4 * q, v.x);
            if (v.y) atomicAdd(gh1 + 4 * q + 1, v.y);
            if (v.z) atomicAdd(gh1 + 4 * q + 2, v.z);
            if (v.w) atomicAdd(gh1 + 4 * q + 3, v.w);
        }
        group_barrier(unit_bar, cpu, gen_unit, wg);

        // ---- 2. the list's masses and histogram, then the cut ---------------
        if (tid == 0) {
            // the barrier's acquire made the other blocks' writes visible to this
            // thread; the proxy fences hand them, and this block's own generic
            // accesses of the ring, over to the bulk copies
            asm volatile("fence.proxy.async.global;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            const uint32_t mbytes = static_cast<uint32_t>((F + 3) / 4 * 16);
            const uint32_t bar = smem_u32(&sh.load_bar);
            mbar_arrive_expect_tx(bar, mbytes + kL1Stride * 4);
            if (mbytes) bulk_load(smem_u32(s_mass), f.mass + static_cast<size_t>(u) * f.ld, mbytes, bar);
            bulk_load(smem_u32(s_h1), gh1, kL1Stride * 4, bar);
        }
        mbar_wait_g(smem_u32(&sh.load_bar), 0u, wg);
        {
            // level-1 cut: thread t owns bins (top_t - 27, top_t] from the top
            const int top = kL1Bins - 1 - tid * kL1Per;
            unsigned long long mine = 0ull;
#pragma unroll
            for (int i = 0; i < kL1Per; ++i) mine += top - i >= 0 ? s_h1[top - i] : 0u;
            unsigned long long total;
            unsigned long long acc = fused_excl_scan(mine, sh.scan64, total);
            if (acc < target && acc + mine >= target) {
                for (int i = 0; i < kL1Per; ++i) {
                    const int bn = top - i;
                    if (bn < 0) break;
                    const uint32_t hv = s_h1[bn];
                    if (acc + hv >= target) {
                        sh.lo = l1_lo(bn);
                        sh.hi = l1_hi(bn);
                        sh.above = acc;
                        sh.found = 1;
                        break;
                    }
                    acc += hv;
                }
            }
        }
        __syncthreads();
        const int nstripe = (F + kThreads - 1) / kThreads;
        const int nq = (F + 3) / 4;                    // groups of 4 masses (one 16-byte load)
        const uint4 *m4 = reinterpret_cast<const uint4 *>(s_mass);
        if (sh.found) {
            // the crossing bin's pages: counted, then written at scanned places
            const uint32_t lo = sh.lo, hi = sh.hi;
            auto in_bin = [&](uint32_t x, int p) { return p < F && x >= lo && x < hi; };
            uint32_t cnt = 0u;
            for (int q = tid; q < nq; q += kThreads) {
                const uint4 v = m4[q];
                cnt += in_bin(v.x, 4 * q) + in_bin(v.y, 4 * q + 1) + in_bin(v.z, 4 * q + 2) + in_bin(v.w, 4 * q + 3);
            }
            uint32_t ntot;
            uint32_t pos = fused_excl_scan(cnt, sh.scan32, ntot);
            if (cnt) {
                for (int q = tid; q < nq; q += kThreads) {
                    const uint4 v = m4[q];
                    const uint32_t xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (in_bin(xv[i], 4 * q + i)) {
                            if (pos < static_cast<uint32_t>(kCand)) s_cand[pos] = xv[i];
                            ++pos;
                        }
                }
            }
            if (tid == 0) sh.ncand = static_cast<int>(ntot);
            __syncthreads();
            const int nc = sh.ncand;
            if (nc <= kCand) {
                if (warp == 0) {
                    uint32_t l2 = lo, h2 = hi;
                    unsigned long long above = sh.above;
                    warp_refine(s_cand, nc, s_h2, kRuleCoverage, target, l2, h2, above);
                    if (lane == 0) {
                        sh.lo = l2;
                        sh.hi = h2;
                        sh.above = above;
                    }
                }
                __syncthreads();
            } else {
                // a crowded crossing bin (many equal masses): 256-bin levels
                // over all of the list's pages
                for (int pass = 0; sh.hi - sh.lo > 1u && pass < 6; ++pass) {
                    const uint32_t plo = sh.lo, phi = sh.hi;
                    int shift, nb;
                    refine_bins(plo, phi, shift, nb);
                    for (int i = tid; i < kL2Bins; i += kThreads) s_h2[i] = 0u;
                    __syncthreads();
                    for (int k = 0; k < nstripe; ++k) {
                        const int p = k * kThreads + tid;
                        const uint32_t x = p < F ? s_mass[p] : 0u;
                        hist_add_warp(s_h2, (x - plo) >> shift, to_fx(x), p < F && x >= plo && x < phi);
                    }
                    __syncthreads();
                    if (warp == 0) {
                        uint32_t nlo = plo, nhi = phi;
                        unsigned long long above = sh.above;
                        warp_pick_bin([&](int bn) { return s_h2[bn]; }, nb, shift, target, nlo, nhi, above);
                        if (lane == 0) {
                            sh.lo = nlo;
                            sh.hi = nhi;
                            sh.above = above;
                        }
                    }
                    __syncthreads();
                }
            }
            if (tid == 0) {
                if (sh.hi - sh.lo > 1u) raise_status(a.status, kDevBadLen);     // cannot happen
                const uint32_t cfx = to_fx(sh.lo);             // > 0: it carried the crossing
                const uint32_t d = static_cast<uint32_t>(target - sh.above);
                sh.cut = sh.lo;
                sh.need = d / cfx + (d % cfx != 0u ? 1u : 0u);
            }
        } else if (tid == 0) {                                 // total < gamma: keep all
            sh.cut = 0u;
            sh.need = 0xFFFFFFFFu;
        }
        __syncthreads();

        // ---- 3. this run's kept pages at their places in the list -----------
        const uint32_t cut = sh.cut, need = sh.need;
        // pages above / at the cut before this run and in the whole list
        unsigned long long cnt = 0ull;                 // 16-bit fields: gt before, eq before, gt, eq
        for (int q = tid; q < nq; q += kThreads) {
            const uint4 v = m4[q];
            const uint32_t xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int p = 4 * q + i;
                if (p < F) {
                    const unsigned long long gt = xv[i] > cut, eq = xv[i] == cut;
                    cnt += (p < P0 ? gt | (eq << 16) : 0ull) | (gt << 32) | (eq << 48);
                }
            }
        }
        // this thread's own pages: above / at the cut
        uint32_t gtm = 0u, eqm = 0u, ng = 0u, ne = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (p4 + i < P1) {
                const uint32_t x = s_mass[p4 + i];
                if (x > cut) {
                    gtm |= 1u << i;
                    ++ng;
                } else if (x == cut) {
                    eqm |= 1u << i;
                    ++ne;
                }
            }
        }
        unsigned long long tot;
        fused_excl_scan(cnt, sh.scan64, tot);
        uint32_t tot2;
        const uint32_t pre = fused_excl_scan(ng | (ne << 16), sh.scan32, tot2);
        const uint32_t gt_before = static_cast<uint32_t>(tot & 0xFFFFu);
        const uint32_t eq_before = static_cast<uint32_t>((tot >> 16) & 0xFFFFu);
        const uint32_t gt_all = static_cast<uint32_t>((tot >> 32) & 0xFFFFu);
        const uint32_t eq_all = static_cast<uint32_t>(tot >> 48);
        int32_t *out = f.lists + static_cast<size_t>(u) * mp;
        uint32_t gb = gt_before + (pre & 0xFFFFu), eb = eq_before + (pre >> 16);
        bool badp = false;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool g = gtm >> i & 1u, e = eqm >> i & 1u;
            if (g || (e && eb < need)) {
                badp |= pref[i] < 0 || pref[i] >= a.num_pages;
                out[gb + min(eb, need)] = pref[i];
            }
            gb += g;
            eb += e;
        }
        if (badp) raise_status(a.status, kDevBadPage);
        if (tid == 0) {
            const int len = static_cast<int>(gt_all + min(eq_all, need)) + (tail != 0);
            if (c == cpu - 1 && tail) out[len - 1] = __ldg(f.page_table + static_cast<size_t>(r) * mp + F);
            if (c == 0) f.lengths[u] = len;
        }
    }

    // ---- every block: the lists and lengths of all lists are written ----------
    if (!f.dense) {
        group_barrier(grid_bar, static_cast<uint32_t>(nblk), gen_grid, wg);
        if (selb) {                                // every block of the list has read its histogram
            uint32_t *gh1 = f.l1hist + static_cast<size_t>(u) * kL1Stride;
            for (int i = c * kL1Stride / cpu + tid; i < (c + 1) * kL1Stride / cpu; i += kThreads) gh1[i] = 0u;
        }
    }

    // ---- plan (warp 0): list lengths and offsets -----------------------------
    if (warp == 0) {
        int len_l[kFusedUnitPer];
#pragma unroll
        for (int k = 0; k < kFusedUnitPer; ++k) {
            const int uu = lane + 32 * k;
            len_l[k] = 0;
            if (uu < U) {
                int Fu, tu;
                request_pages(__ldg(a.seq_lens + uu / a.hkv), mp, Fu, tu);
                s_utail[uu] = tu;
                if (f.dense) {
                    len_l[k] = Fu + (tu != 0);
                    if (b == 0) f.lengths[uu] = len_l[k];
                } else {
                    const int len = __ldcg(f.lengths + uu);          // written in this launch
                    len_l[k] = len < 0 ? 0 : (len > mp ? mp : len);
                }
            }
        }
        int base = 0;
#pragma unroll
        for (int k = 0; k < kFusedUnitPer; ++k) {
            int tk;
            const int ex = warp_excl_scan(len_l[k], tk);
            const int uu = lane + 32 * k;
            if (uu < U) s_off[uu] = base + ex;
            base += tk;
        }
        if (lane == 0) s_off[U] = base;
    }
    __syncthreads();

    // ---- attention over the lists (k_attend's plan and data path) -------------
    const long long W = s_off[U];
    const long long n = min(static_cast<long long>(nblk), W);
    const long long g0 = b < n ? b * W / n : 0;
    const long long g1 = b < n ? (b + 1) * W / n : 0;
    const int hkv = a.hkv;

    if (warp == kConsumerWarps) {
        // the selection wrote the ring through the generic proxy; the TMA
        // loads write it through the asynchronous one
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const bool dense = f.dense != 0;
        attend_produce(sm, stage, &tmap_k, &tmap_v, a, g0, g1, wg, [&](long long k, int &uu, int &ntok, int &pid) {
            int lo = 0, hi = U;                     // largest list uu with s_off[uu] <= k
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (s_off[mid] <= k) lo = mid; else hi = mid;
            }
            uu = lo;
            const int i = static_cast<int>(k - s_off[uu]);
            const int len = s_off[uu + 1] - s_off[uu];
            if (dense) {                            // entry i is logical page i; the output list is written here
                pid = __ldg(f.page_table + static_cast<size_t>(uu / hkv) * mp + i);
                f.lists[static_cast<size_t>(uu) * mp + i] = pid;
            } else {                                // written by this launch's selection
                pid = __ldcg(f.lists + static_cast<size_t>(uu) * mp + i);
            }
            ntok = (s_utail[uu] && i == len - 1) ? s_utail[uu] : kPageSize;
        });
        return;
    }
    attend_consume(sm, stage, s_off, U, W, n, g0, g1, a, wg);
    // after a give-up, the bulk copy of the selection may still be in flight
    if (selb && tid == 0 && guard_failed(wg)) mbar_drain(smem_u32(&sh.load_bar), 0u, globaltimer() + kDrainLimitNs);
}

static size_t select_attend_smem(int units)
{
    return attend_smem_bytes<kFusedSlots, kFusedWarps>(units) + sizeof(int) * static_cast<size_t>(units);
}

bool select_attend_fits(int units, int max_pages, int blocks)
{
    if (units < 1 || units > kFusedMaxUnits || blocks > kFusedMaxBlocks || blocks < units) return false;
    const int cpu = blocks / units;
    const int nch = (max_pages + kScoreChunk - 1) / kScoreChunk;
    if ((nch + cpu - 1) / cpu > kFusedChunks) return false;
    // every block of the grid must be resident at once (the launch has
    // barriers): checked once per device at the largest shared-memory size
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    static std::atomic<int> resident[64];          // 0 unknown, 1 fits, 2 does not
    int known = resident[dev].load(std::memory_order_relaxed);
    if (known == 0) {
        static std::atomic<int> seen[64];
        const size_t smem = select_attend_smem(kFusedMaxUnits);
        int per_sm = 0;
        const bool ok =
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
            raise_smem_limit(k_select_attend<kFusedSlots, kFusedWarps>, smem, seen) == cudaSuccess &&
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_select_attend<kFusedSlots, kFusedWarps>,
                                                          kFusedThreads, smem) == cudaSuccess &&
            per_sm >= kBlocksPerSm && blocks <= sms * kBlocksPerSm;
        known = ok ? 1 : 2;
        resident[dev].store(known, std::memory_order_relaxed);
    }
    return known == 1;
}

cudaError_t launch_select_attend(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                 const FusedArgs &args, int blocks, cudaStream_t stream)
{
    const size_t smem = select_attend_smem(args.at.units);
    static std::atomic<int> seen[64];
    cudaError_t e = raise_smem_limit(k_select_attend<kFusedSlots, kFusedWarps>, smem, seen);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_select_attend<kFusedSlots, kFusedWarps>, dim3(blocks), dim3(kFusedThreads), smem,
                      stream, tmap_k, tmap_v, args);
}

}  // namespace moira
