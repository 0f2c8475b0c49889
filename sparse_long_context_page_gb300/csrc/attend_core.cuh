// Device code shared by the two attention kernels: k_attend (lists from a
// caller or from moira_select) and k_select_attend (the selection and the
// attention of one layer in one launch).  Both take a fixed grid, lay the
// lists end to end, give block b the page range [b*W/n, (b+1)*W/n), stream the
// pages through a TMA ring with one producer warp and NW consumer warps, and
// merge the partials of a list split over several blocks by log-sum-exp
// ("MOIRA: Mass-Oriented Indexing with Ragged Attention for Long-Context
// Decoding", abstract: self-planning ragged attention; FlashDecoding,
// "Faster Flash Decoding" section 2: parallel along the sequence).
//
// Data path per block:
//   the producer looks up a batch of 32 list entries while it issues the
//   previous batch, and issues 2-D TMA tensor loads of each kept page's K and
//   V blocks (16 tokens x 128 dims bf16 = 4 KB each, two 128-byte-swizzled
//   boxes per block) into the ring, tracked by mbarriers; with NW consumer
//   warps, warp w takes pages w, w+NW, ... of the block's range, so each ring
//   slot has one consumer.  The G = 4 query heads of the KV head share every
//   page load:
//     S^T[h][t] = q_h . k_t   : mma.m16n8k16, A = q (rows 0-3 and 4-7 both
//                               hold the 4 heads), B = K^T via ldmatrix
//     O^T[d][n] += V^T P^T    : mma.m16n8k16, A = V^T via ldmatrix.trans,
//                               B columns 0-3 = bf16(P), columns 4-7 = the
//                               bf16 residual P - bf16(P), so P enters the
//                               product with ~16 significant bits
//   with an fp32 online softmax in the log2 domain.
// Merges: a list on at most flat_merge_max() blocks is one group: its last
// block copies all its partials into its own stage ring, idle by then, with
// one bulk copy and merges them there.  Longer lists merge in two levels: the
// last block to finish in each group of 12 consecutive blocks merges the
// group, and the last group to finish writes the output.  Arrival counters
// reset themselves; a list held by one block is written by that block.
#pragma once

#include "moira_device.cuh"
#include "moira_launch.h"

namespace moira {

constexpr int kSlotBytes = 2 * kPageSize * kHeadDim * 2;          // K + V block, 8 KB
constexpr int kHalfBox = kPageSize * 64 * 2;                        // 16 rows x 128 B
constexpr int kBlocksPerSm = 2;
// Two block shapes, both 2 per SM.  Few lists (a small batch, each list
// spread over many blocks, merges on the critical path): 4 consumer warps and
// a 12-slot ring, whose one-level merge reaches lists on 47 blocks.  Many
// lists (short merges; the consumer warps set the rate): 5 consumer warps and
// a 10-slot ring.  The slot count is a multiple of the consumer warps.
constexpr int kFewSlots = 12, kFewWarps = 4;
constexpr int kManySlots = 10, kManyWarps = 5;
constexpr int kManyUnits = 64;            // lists per launch from which the second shape runs

template <int NS, int NW>
struct AttendSmem {
    float co[NW][kGroup][kHeadDim];
    float cm[NW][kGroup];
    float cl[NW][kGroup];
    unsigned long long full[NS];
    unsigned long long empty[NS];
    int2 meta[NS];            // (unit, valid tokens; 0 = skip)
    int flag;
    int abort;                // the block's WaitGuard flag
    int merge_pending;        // a merge bulk copy was issued and not seen to land
    int pad;
    unsigned long long mrg;   // one-level merge: the bulk copy of a list's partials
};

template <int NS, int NW>
__host__ __device__ inline size_t attend_smem_bytes(int units)
{
    return 1024 + static_cast<size_t>(NS) * kSlotBytes + sizeof(AttendSmem<NS, NW>) +
           sizeof(int) * static_cast<size_t>(units + 1);
}

constexpr int kLenCache = 4;              // list lengths per thread kept in registers by the plan scan
constexpr int kMergeSpan = 12;            // blocks per first-level merge group
constexpr int kMergeBatch = 12;           // partials loaded together in a merge
// A list spread over at most this many blocks merges in one level: its last
// block copies all its partials into its stage ring (idle by then).
template <int NS>
__host__ __device__ constexpr int flat_merge_max() { return NS * kSlotBytes / (kPartFloats * 4); }

// Online log-sum-exp merge of `count` partials stored at slots first,
// first + stride, ... for this thread's head h and dims d0..d0+3: returns the
// merged (max, sum, unnormalised o).  All loads of a batch are in flight
// together; L2-only loads because other blocks wrote the partials.
__device__ __forceinline__ void merge_partials(const float *partials, int first, int stride,
                                               int count, int h, int d0, float &Mout,
                                               float &Lout, float4 &Oout)
{
    float Mrun = -INFINITY, la = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < count; k0 += kMergeBatch) {
        float mv[kMergeBatch], lv[kMergeBatch];
        float4 ov[kMergeBatch];
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            mv[k] = -INFINITY;
            lv[k] = 0.f;
            ov[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k0 + k < count) {
                const float *pp = partials + static_cast<size_t>(first + (k0 + k) * stride) * kPartFloats;
                mv[k] = __ldcg(pp + h);
                lv[k] = __ldcg(pp + kGroup + h);
                ov[k] = __ldcg(reinterpret_cast<const float4 *>(pp + 2 * kGroup + h * kHeadDim + d0));
            }
        }
        float mb = Mrun;
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) mb = fmaxf(mb, mv[k]);
        const float ms = mb == -INFINITY ? 0.f : mb;
        const float sc = exp2f(Mrun - ms);
        acc.x *= sc; acc.y *= sc; acc.z *= sc; acc.w *= sc;
        la *= sc;
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            const float e = exp2f(mv[k] - ms);
            acc.x += e * ov[k].x; acc.y += e * ov[k].y; acc.z += e * ov[k].z; acc.w += e * ov[k].w;
            la += e * lv[k];
        }
        Mrun = mb;
    }
    Mout = Mrun;
    Lout = la;
    Oout = acc;
}

// Largest b with floor(b*W/n) <= g: the block whose range holds page g.
__device__ __forceinline__ int block_of(long long g, long long W, long long n)
{
    return static_cast<int>(((g + 1) * n - 1) / W);
}

// Named barrier of the NW consumer warps (the producer warp never joins it).
template <int NW>
__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

__device__ __forceinline__ float *out_row(const AttendArgs &a, int u, int h, int d0)
{
    const int r = u / a.hkv, j = u % a.hkv;
    return a.out + (static_cast<size_t>(r) * a.hq + j * kGroup + h) * kHeadDim + d0;
}

// How list u is spread over the blocks: blocks bfirst..blast hold its pages;
// block b's merge group starts at gfirst and has gn members; the list has
// ngroups groups.  A list on at most flat_max blocks is one group.
struct ListSplit {
    int bfirst, blast, gfirst, gn, ngroups;
};

__device__ __forceinline__ ListSplit list_split(const int *s_off, int u, int b, long long W, long long n,
                                                int flat_max)
{
    ListSplit ls;
    ls.bfirst = block_of(s_off[u], W, n);
    ls.blast = block_of(static_cast<long long>(s_off[u + 1]) - 1, W, n);
    if (ls.blast - ls.bfirst + 1 <= flat_max) {
        ls.gfirst = ls.bfirst;
        ls.gn = ls.blast - ls.bfirst + 1;
        ls.ngroups = 1;
        return ls;
    }
    ls.gfirst = ls.bfirst + (b - ls.bfirst) / kMergeSpan * kMergeSpan;
    ls.gn = min(kMergeSpan, ls.blast - ls.gfirst + 1);
    ls.ngroups = (ls.blast - ls.bfirst) / kMergeSpan + 1;
    return ls;
}

// Merge of `count` partials that sit contiguously in shared memory, for this
// thread's head h and dims d0..d0+3 (two passes: the maximum, then the sums).
__device__ __forceinline__ void merge_partials_smem(const float *pp, int count, int h, int d0, float &Mout,
                                                    float &Lout, float4 &Oout)
{
    float mb = -INFINITY;
    for (int k = 0; k < count; ++k) mb = fmaxf(mb, pp[k * kPartFloats + h]);
    const float ms = mb == -INFINITY ? 0.f : mb;
    float la = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < count; ++k) {
        const float *q = pp + k * kPartFloats;
        const float e = exp2f(q[h] - ms);
        const float4 o = *reinterpret_cast<const float4 *>(q + 2 * kGroup + h * kHeadDim + d0);
        acc.x += e * o.x; acc.y += e * o.y; acc.z += e * o.z; acc.w += e * o.w;
        la += e * q[kGroup + h];
    }
    Mout = mb;
    Lout = la;
    Oout = acc;
}

// Where a merge may land its copy of the partials: the block's stage ring.
struct MergeRing {
    uint8_t *ring;
    uint32_t bar;
    uint32_t phase;
    int *pending;             // shared: a copy was issued and its landing not yet seen
};

// Merges after this block's partial of a shared list u is published; prev is
// the value thread 0's arrival atomic on the group counter returned (unused
// for a group of one).  The last block to arrive in a group merges the group
// (into the output when the list has one group); the last group to arrive
// merges the groups into the output.  Called by all NW consumer warps; only
// the first 4 (one per (head, 4 dims)) write.
template <int NW>
__device__ __forceinline__ void resolve_list(const AttendArgs &a, int &flag, int u, const ListSplit ls,
                                             uint32_t prev, int h, int d0, MergeRing &mr, const WaitGuard &wg)
{
    const int tid = threadIdx.x;
    const bool hw = NW == kGroup || tid < kGroup * 32;   // always true with 4 consumer warps
    int mine = 1;
    if (ls.gn > 1) {
        if (tid == 0) flag = (prev == static_cast<uint32_t>(ls.gn - 1)) ? 1 : 0;
        consumer_bar<NW>();
        mine = *const_cast<volatile int *>(&flag);
        consumer_bar<NW>();                                  // every thread has read flag
        if (mine) {
            float gm, gl;
            float4 go;
            if (ls.gn > kMergeBatch) {
                // one bulk copy of the group's partials (consecutive slots) into
                // the idle ring instead of several rounds of L2 loads.  The
                // acquire above made the other blocks' partials visible to this
                // thread; the proxy fences hand them, and the ring's last
                // generic reads, over to the asynchronous copy.
                const uint32_t bytes = static_cast<uint32_t>(ls.gn) * kPartFloats * 4;
                if (tid == 0) {
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    *mr.pending = 1;
                    mbar_arrive_expect_tx(mr.bar, bytes);
                    bulk_load(smem_u32(mr.ring), a.partials + static_cast<size_t>(ls.gfirst + u) * kPartFloats,
                              bytes, mr.bar);
                }
                if (mbar_wait_g(mr.bar, mr.phase, wg) && tid == 0) *mr.pending = 0;
                mr.phase ^= 1u;
                merge_partials_smem(reinterpret_cast<const float *>(mr.ring), ls.gn, h, d0, gm, gl, go);
            } else {
                merge_partials(a.partials, ls.gfirst + u, 1, ls.gn, h, d0, gm, gl, go);
            }
            if (ls.ngroups == 1) {                       // the only group: write the output
                const float inv = gl > 0.f ? 1.f / gl : 0.f;
                if (hw)
                    *reinterpret_cast<float4 *>(out_row(a, u, h, d0)) =
                        make_float4(go.x * inv, go.y * inv, go.z * inv, go.w * inv);
            } else {
                consumer_bar<NW>();                          // the group's first slot is read
                float *gp = a.partials + static_cast<size_t>(ls.gfirst + u) * kPartFloats;
                if (hw) *reinterpret_cast<float4 *>(gp + 2 * kGroup + h * kHeadDim + d0) = go;
                if (hw && (tid & 31) == 0) {
                    gp[h] = gm;
                    gp[kGroup + h] = gl;
                }
            }
            if (tid == 0) a.gcounters[ls.gfirst + u] = 0u;      // ready for the next launch
        }
    }
    if (mine && ls.ngroups > 1) {
        consumer_bar<NW>();                                  // group partial written
        if (tid == 0) {
            const uint32_t p2 = atomic_add_acq_rel_gpu(&a.counters[u], 1u);
            flag = (p2 == static_cast<uint32_t>(ls.ngroups - 1)) ? 1 : 0;
        }
        consumer_bar<NW>();
        const int last = *const_cast<volatile int *>(&flag);
        if (last) {
            float fm, fl;
            float4 fo;
            merge_partials(a.partials, ls.bfirst + u, kMergeSpan, ls.ngroups, h, d0, fm, fl, fo);
            const float inv = fl > 0.f ? 1.f / fl : 0.f;
            if (hw)
                *reinterpret_cast<float4 *>(out_row(a, u, h, d0)) =
                    make_float4(fo.x * inv, fo.y * inv, fo.z * inv, fo.w * inv);
            if (tid == 0) a.counters[u] = 0u;            // ready for the next launch
        }
    }
    consumer_bar<NW>();                                      // flag is free again
}

// Set-up shared by the attention kernels: the 1024-aligned stage ring, the
// mbarriers and the wait guard.  Thread 0 initialises; the caller must pass
// a __syncthreads (or a barrier that implies one) before the first use.
template <int kSlots, int kConsumerWarps>
__device__ __forceinline__ void attend_init(AttendSmem<kSlots, kConsumerWarps> &sm, const CUtensorMap *tmap_k,
                                            const CUtensorMap *tmap_v, uint32_t *status)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 1);
        }
        mbar_init(smem_u32(&sm.mrg), 1);
        mbar_fence_init();
        sm.merge_pending = 0;
        WaitGuard wg{&sm.abort, status};
        guard_init(wg);
    }
    if (warp == kConsumerWarps && lane == 0) {
        tma_prefetch_desc(tmap_k);
        tma_prefetch_desc(tmap_v);
    }
}

// The producer warp: lane i resolves entry base+i of a batch of 32 (its list,
// physical id and valid-token count) through lookup(k, u, ntok, pid), called
// only for k < g1.  The next batch's lookups are in flight while the current
// batch's copies are issued, so list reads do not stall the ring; the copies
// are issued by kIssueLanes lanes at once (one page each: at most one lane
// per ring slot), since one lane issuing page after page could not keep the
// ring full.
constexpr int kIssueLanes = 8;
static_assert(kIssueLanes <= kManySlots && kIssueLanes <= kFewSlots && 32 % kIssueLanes == 0,
              "an issue group never holds two pages of one ring slot");
template <int kSlots, int kConsumerWarps, class Lookup>
__device__ __forceinline__ void attend_produce(AttendSmem<kSlots, kConsumerWarps> &sm, uint8_t *stage,
                                               const CUtensorMap *tmap_k, const CUtensorMap *tmap_v,
                                               const AttendArgs &a, long long g0, long long g1,
                                               const WaitGuard &wg, Lookup lookup)
{
    const int lane = threadIdx.x & 31;
    auto look = [&](long long k, int &u, int &ntok, int &pid) {
        u = 0;
        ntok = 0;
        pid = 0;
        if (k < g1) lookup(k, u, ntok, pid);
    };
    // small batches: K/V are read once and must not push the merge partials
    // and list data out of L2
    const uint64_t pol = l2_evict_first();
    int cu, cn, cp;
    look(g0 + lane, cu, cn, cp);
    for (long long base = g0; base < g1; base += 32) {
        int nu, nn, np;
        look(base + 32 + lane, nu, nn, np);
        if (cn > 0 && (cp < 0 || cp >= a.num_pages)) {
            cn = 0;
            raise_status(a.status, kDevBadPage);
        }
        const int cnt = static_cast<int>(min(32LL, g1 - base));
        // kIssueLanes lanes at a time, each filling its own ring slot: entry
        // idx goes to slot idx % kSlots once the slot's previous round
        // (entry idx - kSlots, issued by an earlier group) has been consumed
        for (int q0 = 0; q0 < cnt; q0 += kIssueLanes) {
            if (lane >= q0 && lane < q0 + kIssueLanes && lane < cnt) {
                const long long idx = base + lane - g0;
                const int slot = static_cast<int>(idx % kSlots);
                const uint32_t round = static_cast<uint32_t>(idx / kSlots);
                mbar_wait_g(smem_u32(&sm.empty[slot]), (round & 1u) ^ 1u, wg);
                sm.meta[slot] = make_int2(cu, cn);
                const uint32_t full = smem_u32(&sm.full[slot]);
                if (cn > 0) {
                    const uint32_t dst = smem_u32(stage + slot * kSlotBytes);
                    const int row = (cp * a.hkv + cu % a.hkv) * kPageSize;
                    mbar_arrive_expect_tx(full, kSlotBytes);
                    if constexpr (kConsumerWarps == kFewWarps) {
                        tma_load_2d_hint(dst, tmap_k, 0, row, full, pol);
                        tma_load_2d_hint(dst + kHalfBox, tmap_k, 64, row, full, pol);
                        tma_load_2d_hint(dst + 2 * kHalfBox, tmap_v, 0, row, full, pol);
                        tma_load_2d_hint(dst + 3 * kHalfBox, tmap_v, 64, row, full, pol);
                    } else {
                        tma_load_2d(dst, tmap_k, 0, row, full);
                        tma_load_2d(dst + kHalfBox, tmap_k, 64, row, full);
                        tma_load_2d(dst + 2 * kHalfBox, tmap_v, 0, row, full);
                        tma_load_2d(dst + 3 * kHalfBox, tmap_v, 64, row, full);
                    }
                } else {
                    mbar_arrive(full);
                }
            }
            __syncwarp();
        }
        cu = nu;
        cn = nn;
        cp = np;
    }
}

// The consumer warps over the block's range [g0, g1) of the lists laid end to
// end (s_off: exclusive prefix of the list lengths, s_off[units] = W; n
// active blocks), then the merges.  Writes zeros for empty lists (block 0).
template <int kSlots, int kConsumerWarps>
__device__ __forceinline__ void attend_consume(AttendSmem<kSlots, kConsumerWarps> &sm, uint8_t *stage,
                                               const int *s_off, int units, long long W, long long n,
                                               long long g0, long long g1, const AttendArgs &a,
                                               const WaitGuard &wg)
{
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.x;
#ifdef MOIRA_CTA_TIMES
    // load-balance build: the block's attention work, from its plan to the
    // end of its merges, in %globaltimer ns (0, 0 for a block without work)
    const unsigned long long t_start = globaltimer();
    if (a.cta_times && tid == 0 && g0 >= g1) a.cta_times[2 * b] = a.cta_times[2 * b + 1] = 0ull;
#endif
    // empty lists produce zeros (no block would otherwise touch them)
    if (b == 0) {
        for (int u = 0; u < units; ++u) {
            if (s_off[u + 1] != s_off[u]) continue;
            const int r = u / a.hkv, j = u % a.hkv;
            for (int e = tid; e < kGroup * kHeadDim; e += kConsumerWarps * 32)
                a.out[(static_cast<size_t>(r) * a.hq + j * kGroup) * kHeadDim + e] = 0.f;
        }
    }
    if (g0 >= g1) return;

    // this lane's row head in the S^T fragments and its two output columns
    const int hq_row = (lane >> 2) & 3;
    const int tq = 2 * (lane & 3);
    const int hn0 = (2 * (lane & 3)) & 3;
    const bool lo_lane = lane >= 16;      // holds the bf16 residual column of P
    const float c = a.scale_log2;
    // this thread's (head, 4 dims) in the block result and the merges
    // (a fifth consumer warp reads head 0's slice and writes nothing)
    const bool hw = kConsumerWarps == kGroup || tid < kGroup * 32;
    const int h = hw ? tid >> 5 : 0, d0 = (tid & 31) * 4;
    MergeRing mring{stage, smem_u32(&sm.mrg), 0u, &sm.merge_pending};

    // q fragments of list v (A operand rows 0-7 = heads 0-3 twice, rows 8-15 zero)
    uint32_t aq[8][2];
    auto load_q = [&](int v) {
        const int r = v / a.hkv, j = v % a.hkv;
        const uint16_t *qrow = static_cast<const uint16_t *>(a.q) +
                               (static_cast<size_t>(r) * a.hq + j * kGroup + hq_row) * kHeadDim + tq;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            aq[ks][0] = __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16));
            aq[ks][1] = __ldg(reinterpret_cast<const uint32_t *>(qrow + ks * 16 + 8));
        }
    };

    int u;
    {
        int lo = 0, hi = units;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_off[mid] <= g0) lo = mid; else hi = mid;
        }
        u = lo;                            // s_off[u] <= g0 < s_off[u + 1]: list u is not empty
    }
    load_q(u);

    // The first segment's list may continue in earlier blocks.  When more
    // segments follow, its partial is written at once but its arrival (an
    // acq_rel atomic, whose release half waits for the partial to reach L2)
    // and its merges wait for the block's last segment, so the consumer warps
    // go straight on to the next list.
    int pend_u = -1;

    while (true) {
        const long long seg_lo = max(g0, static_cast<long long>(s_off[u]));
        const long long seg_hi = min(g1, static_cast<long long>(s_off[u + 1]));
        float m_run = -INFINITY, l_run = 0.f;
        float D[8][4];
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) D[mt][0] = D[mt][1] = D[mt][2] = D[mt][3] = 0.f;

        // the next list's q rows (4 heads x 256 B) towards L2 while this segment streams
        if (seg_hi < g1 && warp == 0 && lane < 8) {
            int un = u + 1;
            while (s_off[un + 1] == s_off[un]) ++un;
            const int r = un / a.hkv, j = un % a.hkv;
            const char *qn = reinterpret_cast<const char *>(static_cast<const uint16_t *>(a.q) +
                                                          (static_cast<size_t>(r) * a.hq + j * kGroup) * kHeadDim);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + lane * 128));
        }
        const long long first = seg_lo + ((warp - (seg_lo - g0) % kConsumerWarps + kConsumerWarps) % kConsumerWarps);
        for (long long g = first; g < seg_hi; g += kConsumerWarps) {
            const long long idx = g - g0;
            const int slot = static_cast<int>(idx % kSlots);
            const uint32_t round = static_cast<uint32_t>(idx / kSlots);
            mbar_wait_g(smem_u32(&sm.full[slot]), round & 1u, wg);
            const int ntok = sm.meta[slot].y;
            if (ntok > 0) {
                const uint32_t kb = smem_u32(stage + slot * kSlotBytes);
                const uint32_t vb = kb + 2 * kHalfBox;
                // ---- S^T = q K^T for the 4 heads x 16 tokens ----
                float acc[4][4];
#pragma unroll
                for (int x = 0; x < 4; ++x) acc[x][0] = acc[x][1] = acc[x][2] = acc[x][3] = 0.f;
                {
                    const int t = (lane & 7) + ((lane >> 4) << 3);
                    const int sw = t & 7;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int ch = 2 * ks + ((lane >> 3) & 1);
                        const uint32_t addr = kb + (ch >> 3) * kHalfBox + t * 128 + (((ch & 7) ^ sw) << 4);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(addr, b0, b1, b2, b3);
                        const int par = (ks & 1) * 2;
                        mma_bf16_16816(acc[par], aq[ks][0], 0u, aq[ks][1], 0u, b0, b1);
                        mma_bf16_16816(acc[par + 1], aq[ks][0], 0u, aq[ks][1], 0u, b2, b3);
                    }
                }
                float s[4] = {(acc[0][0] + acc[2][0]) * c, (acc[0][1] + acc[2][1]) * c,
                              (acc[1][0] + acc[3][0]) * c, (acc[1][1] + acc[3][1]) * c};
                const bool tail = ntok < kPageSize;
                if (tail) {
                    if (tq >= ntok) s[0] = -INFINITY;
                    if (tq + 1 >= ntok) s[1] = -INFINITY;
                    if (tq + 8 >= ntok) s[2] = -INFINITY;
                    if (tq + 9 >= ntok) s[3] = -INFINITY;
                }
                float pm = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
                pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 1));
                pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 2));
                const float m_new = fmaxf(m_run, pm);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = exp2f(m_run - m_use);
                float p[4];
#pragma unroll
                for (int x = 0; x < 4; ++x) p[x] = exp2f(s[x] - m_use);
                l_run = l_run * alpha + (p[0] + p[1]) + (p[2] + p[3]);
                m_run = m_new;
                // B operand: columns 0-3 bf16(P), columns 4-7 residual
                uint32_t bp0, bp1;
                {
                    uint32_t hb4[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const uint32_t hb = f32_to_bf16_rne(p[x]);
                        hb4[x] = lo_lane ? f32_to_bf16_rne(p[x] - __uint_as_float(hb << 16)) : hb;
                    }
                    bp0 = hb4[0] | (hb4[1] << 16);
                    bp1 = hb4[2] | (hb4[3] << 16);
                }
                // rescale the running O^T columns (heads hn0, hn0+1)
                const float al0 = __shfl_sync(0xffffffffu, alpha, 4 * hn0);
                const float al1 = __shfl_sync(0xffffffffu, alpha, 4 * (hn0 + 1));
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        D[mt][0] *= al0;
                        D[mt][1] *= al1;
                        D[mt][2] *= al0;
                        D[mt][3] *= al1;
                    }
                }
                // ---- O^T += V^T P^T ----
                uint32_t msk01 = 0xFFFFFFFFu, msk23 = 0xFFFFFFFFu;
                if (tail) {
                    msk01 = (tq < ntok ? 0x0000FFFFu : 0u) | (tq + 1 < ntok ? 0xFFFF0000u : 0u);
                    msk23 = (tq + 8 < ntok ? 0x0000FFFFu : 0u) | (tq + 9 < ntok ? 0xFFFF0000u : 0u);
                }
                {
                    const int mi = lane >> 3;
                    const int t = (lane & 7) + ((mi >> 1) << 3);
                    const int sw = t & 7;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        const int ch = 2 * mt + (mi & 1);
                        const uint32_t addr = vb + (ch >> 3) * kHalfBox + t * 128 + (((ch & 7) ^ sw) << 4);
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_trans(addr, a0, a1, a2, a3);
                        mma_bf16_16816(D[mt], a0 & msk01, a1 & msk01, a2 & msk23, a3 & msk23, bp0, bp1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.empty[slot]));
        }

        // the next non-empty list of this block: its q loads overlap the
        // combine below (the current q is no longer needed)
        const bool more = seg_hi < g1;
        int un = u + 1;
        if (more) {
            while (s_off[un + 1] == s_off[un]) ++un;
            load_q(un);
        }

        // ---- warp result -> shared memory ----
        float lsum = l_run + __shfl_xor_sync(0xffffffffu, l_run, 1);
        lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float v = D[mt][x] + __shfl_xor_sync(0xffffffffu, D[mt][x], 2);
                if ((lane & 3) < 2) {
                    const int hh = 2 * (lane & 3) + (x & 1);
                    const int d = 16 * mt + (lane >> 2) + (x >= 2 ? 8 : 0);
                    sm.co[warp][hh][d] = v;
                }
            }
        }
        if (lane < 16 && (lane & 3) == 0) {
            sm.cm[warp][lane >> 2] = m_run;
            sm.cl[warp][lane >> 2] = lsum;
        }
        consumer_bar<kConsumerWarps>();

        // ---- block result: thread -> (head, 4 dims) ----
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.cm[w][h]);
        const float Ms = M == -INFINITY ? 0.f : M;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        float Lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float e = exp2f(sm.cm[w][h] - Ms);
            const float4 v = *reinterpret_cast<const float4 *>(&sm.co[w][h][d0]);
            o.x += e * v.x; o.y += e * v.y; o.z += e * v.z; o.w += e * v.w;
            Lsum += e * sm.cl[w][h];
        }
        const ListSplit ls = list_split(s_off, u, b, W, n, flat_merge_max<kSlots>());
        if (ls.bfirst == ls.blast) {
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
            if (hw)
                *reinterpret_cast<float4 *>(out_row(a, u, h, d0)) =
                    make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv);
        } else {
            // this block's partial of list u -> slot b + u, then its arrival
            float *part = a.partials + static_cast<size_t>(b + u) * kPartFloats;
            if (hw) *reinterpret_cast<float4 *>(part + 2 * kGroup + h * kHeadDim + d0) = o;
            if (hw && (tid & 31) == 0) {
                part[h] = M;
                part[kGroup + h] = Lsum;
            }
            if (more) {                    // first segment: arrival and merges after the last one
                pend_u = u;
            } else {
                // the CTA barrier makes every thread's partial visible to thread 0,
                // whose acq_rel atomic publishes it and acquires the others
                consumer_bar<kConsumerWarps>();
                uint32_t prev = 0u;
                if (ls.gn > 1 && tid == 0) prev = atomic_add_acq_rel_gpu(&a.gcounters[ls.gfirst + u], 1u);
                resolve_list<kConsumerWarps>(a, sm.flag, u, ls, prev, h, d0, mring, wg);
            }
        }
        consumer_bar<kConsumerWarps>();    // sm.co / cm / cl are reused by the next segment
        if (!more) break;
        u = un;
    }
    if (pend_u >= 0) {
        // its partial was written before the segment's closing barrier
        const ListSplit ls = list_split(s_off, pend_u, b, W, n, flat_merge_max<kSlots>());
        uint32_t prev = 0u;
        if (ls.gn > 1 && tid == 0) prev = atomic_add_acq_rel_gpu(&a.gcounters[ls.gfirst + pend_u], 1u);
        resolve_list<kConsumerWarps>(a, sm.flag, pend_u, ls, prev, h, d0, mring, wg);
    }

    // after a give-up, let the copies still in flight land before the block
    // exits (their landing is what the skipped waits were for)
    if (tid == 0 && guard_failed(wg)) {
        const uint64_t deadline = globaltimer() + kDrainLimitNs;
        const long long N = g1 - g0;
        for (int s = 0; s < kSlots && s < N; ++s) {
            const long long last = N - 1 - ((N - 1 - s) % kSlots);        // last entry on slot s
            mbar_drain(smem_u32(&sm.full[s]), static_cast<uint32_t>(last / kSlots) & 1u, deadline);
        }
        if (sm.merge_pending) mbar_drain(smem_u32(&sm.mrg), mring.phase ^ 1u, deadline);
    }
#ifdef MOIRA_CTA_TIMES
    consumer_bar<kConsumerWarps>();
    if (a.cta_times && tid == 0) {
        a.cta_times[2 * b] = t_start;
        a.cta_times[2 * b + 1] = globaltimer();
    }
#endif
}

}  // namespace moira
