// Device-side building blocks shared by the MOIRA kernels (sm_103a).
// Inline PTX for the Blackwell data path: mbarrier-tracked TMA tensor loads,
// ldmatrix and warp-level bf16 tensor-core MMA.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moira {

constexpr int kHeadDim = 128;           // d
constexpr int kPageSize = 16;           // S
constexpr int kGroup = 4;               // G = Hq / Hkv
constexpr int kMaxPagesPerSeq = 16384;      // 256k tokens: 16 stripes of 1024 pages per selection block
constexpr int kMaxUnits = 4096;

constexpr uint32_t kDevBadPage = 0x1u;
constexpr uint32_t kDevBadLen = 0x2u;
constexpr uint32_t kDevTimeout = 0x4u;

// ---- page-summary formats ----------------------------------------------------
// kSummBf16 : bf16 [P][Hkv][d], the mean key rounded to bf16.
// kSummQ8 / kSummQ2 : one record per physical page, the mean key in 8 or 2
//   bits per element (symmetric mid-rise: value = (code + 1/2) * step).  The
//   KV heads are stored in groups of gh = min(Hkv, 4) consecutive heads, one
//   group after another, each group
//     bytes [0, gh*cb)            codes, head jj of the group at [jj*cb, (jj+1)*cb),
//                                 cb = d * bits / 8; Q8: byte i = int8 code of
//                                 element i; Q2: element i in bits 2*(i%4) ..
//                                 2*(i%4)+1 of byte i/4, holding code + 2 (0..3)
//     bytes [gh*cb, gh*cb + 4*gh) fp32 step of each head of the group
//     then zeros up to gh*cb + 16
//   so one group (the heads one score item reads) is one contiguous copy.
constexpr int kSummBf16 = 0;
constexpr int kSummQ8 = 1;
constexpr int kSummQ2 = 2;
constexpr int kSummGroup = 4;           // KV heads per low-bit group

__host__ __device__ constexpr int summ_bits(int fmt) { return fmt == kSummQ8 ? 8 : (fmt == kSummQ2 ? 2 : 16); }
__host__ __device__ constexpr int lowbit_code_bytes(int bits) { return kHeadDim * bits / 8; }
__host__ __device__ constexpr int lowbit_group_heads(int hkv) { return hkv < kSummGroup ? hkv : kSummGroup; }
// Bytes of one low-bit head group: codes, gh fp32 steps, padding to 16 bytes.
__host__ __device__ constexpr int lowbit_group_bytes(int bits, int hkv)
{
    return lowbit_group_heads(hkv) * lowbit_code_bytes(bits) + 16;
}
// Bytes of one physical page's summaries (all KV heads; Hkv in {1, 2, 4, 8}).
__host__ __device__ constexpr int summ_page_bytes(int fmt, int hkv)
{
    return fmt == kSummBf16 ? hkv * kHeadDim * 2
                            : (hkv / lowbit_group_heads(hkv)) * lowbit_group_bytes(summ_bits(fmt), hkv);
}

// A bounded device wait gives up after this long (ns of %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---- workspace layout ------------------------------------------------------
// [0, 256)                    : uint32 status word (+ padding)
// counters                    : uint32 [kMaxUnits]  per-list merge arrival counters
// group counters              : uint32 [n_blocks + units] per-group arrival counters
// weights                     : fp32 [batch][Hq][ld]   chunk-relative page weights 2^(s - M_c)
// chunk stats                 : fp32 [batch][Hq][ldc]  (M_c, sum 2^(s - M_c)) per 32-page chunk
// partials                    : fp32 [n_blocks + units][kPartFloats]
constexpr int kScoreChunk = 32;                    // pages per score block
constexpr int kPartFloats = 2 * kGroup + kGroup * kHeadDim;   // m[G], l[G], o[G][d]

// Row strides: weights rows padded to 32 pages, chunk-stat rows to 16 bytes.
__host__ __device__ inline int weights_ld(int max_pages) { return (max_pages + 31) / 32 * 32; }
__host__ __device__ inline int chunks_ld(int max_pages)
{
    const int nch = (max_pages + kScoreChunk - 1) / kScoreChunk;
    return (2 * nch + 3) / 4 * 4;
}

// Fused selection + attention (k_select_attend, small batches) adds:
// barriers                    : uint32 [kFusedMaxUnits + 1][kBarWords] one barrier per list, then the grid's
// level-1 histograms          : uint32 [fu][kL1Stride]       per list, fixed-point mass per bin
// page masses                 : uint32 [fu][ld]              per list, the fp32 bit pattern of every page's mass
// with fu = min(units, kFusedMaxUnits).  The barriers and histograms start at
// zero (moira_workspace_init) and every launch leaves them at zero.
constexpr int kFusedMaxUnits = 63;                 // lists per launch of the fused kernel
constexpr uint32_t kKeyLo = 95u << 7;               // level-1 bins: see l1_bin()
constexpr int kL1Bins = (16384 - static_cast<int>(kKeyLo)) + 1;     // 4225
constexpr int kL1Stride = (kL1Bins + 3) / 4 * 4;    // 4228: rows of whole 16-byte units
constexpr int kL2Bins = 256;
constexpr int kCand = 2048;                         // crossing-bin pages refined by one warp
constexpr int kBarWords = 32;                       // uint32 words per inter-block barrier (128 B)

struct WsLayout {
    size_t status, counters, gcounters, scores, chunks, partials;
    size_t fbars, fl1, fmass, total;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int batch, int hq, int max_pages, int units, int blocks)
{
    WsLayout w;
    size_t o = 0;
    w.status = o;   o += 256;
    w.counters = o; o = align_up(o + sizeof(uint32_t) * kMaxUnits, 256);
    w.gcounters = o; o = align_up(o + sizeof(uint32_t) * (size_t)(blocks + units), 256);
    w.scores = o;   o = align_up(o + sizeof(float) * (size_t)batch * hq * weights_ld(max_pages), 256);
    w.chunks = o;   o = align_up(o + sizeof(float) * (size_t)batch * hq * chunks_ld(max_pages), 256);
    w.partials = o; o = align_up(o + sizeof(float) * kPartFloats * (size_t)(blocks + units), 256);
    const size_t fu = units < kFusedMaxUnits ? (size_t)units : (size_t)kFusedMaxUnits;
    w.fbars = o;    o = align_up(o + sizeof(uint32_t) * kBarWords * (size_t)(kFusedMaxUnits + 1), 256);
    w.fl1 = o;      o = align_up(o + sizeof(uint32_t) * kL1Stride * fu, 256);
    w.fmass = o;    o = align_up(o + sizeof(uint32_t) * fu * (size_t)weights_ld(max_pages), 256);
    w.total = o;
    return w;
}

// ---- small helpers -----------------------------------------------------------
__device__ __forceinline__ void raise_status(uint32_t *status, uint32_t bits) { atomicOr(status, bits); }

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// fp32 -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float f)
{
    uint32_t u = __float_as_uint(f);
    return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Atomic add at GPU scope with acquire-release semantics: the writes this
// thread has observed (e.g. a CTA's writes made visible to it by a CTA
// barrier) are released before the add, and the caller acquires what earlier
// releasers published.  Returns the previous value.
__device__ __forceinline__ uint32_t atomic_add_acq_rel_gpu(uint32_t *addr, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// ---- mbarrier ------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `parity` to complete, giving up after `limit_ns`.
// Returns false on timeout.  The kernels wait through WaitGuard (below); this
// plain form serves the diagnostic of a single wait.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// ---- bounded waits, given up once per launch ------------------------------------
// Every wait of a kernel goes through the block's WaitGuard: a flag in shared
// memory that the block sets when one of its waits runs out, and that starts
// set when the status word already holds MOIRA_DEV_TIMEOUT (a step whose
// earlier launch timed out waits no more).  A wait checks the flag while it
// spins; once the flag is set, every later wait of the block makes one
// attempt and gives up.  So a copy that never lands costs one wait limit per
// launch instead of one per wait, and the block still follows its normal
// control flow (all loops are bounded by sizes, never by the data waited for).
struct WaitGuard {
    int *flag;              // shared memory, one per block
    uint32_t *status;       // device status word (MOIRA_DEV_* bits)
};

__device__ __forceinline__ bool guard_failed(const WaitGuard &g)
{
    return *const_cast<volatile int *>(g.flag) != 0;
}

__device__ __forceinline__ void guard_fail(const WaitGuard &g)
{
    *const_cast<volatile int *>(g.flag) = 1;
    atomicOr(g.status, kDevTimeout);
}

// Thread 0 sets the flag from the status word before the block's first
// barrier; the word may be stale, which only delays the give-up.
__device__ __forceinline__ void guard_init(const WaitGuard &g)
{
    *g.flag = (__ldcg(g.status) & kDevTimeout) ? 1 : 0;
}

__device__ __forceinline__ bool mbar_wait_g(uint32_t bar, uint32_t parity, const WaitGuard &g,
                                            uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    if (!guard_failed(g)) {
        const uint64_t t0 = globaltimer();
        while (true) {
#pragma unroll 1
            for (int i = 0; i < 32; ++i)
                if (mbar_try_wait(bar, parity)) return true;
            if (guard_failed(g)) break;
            if (globaltimer() - t0 > limit_ns) {
                guard_fail(g);
                break;
            }
        }
    }
    return mbar_try_wait(bar, parity);
}

// After a give-up, copies the block issued may still be in flight towards its
// shared memory; before the block exits, wait for the phase of `parity` of
// every such barrier, at most until `deadline` (globaltimer ns) in all.
constexpr uint64_t kDrainLimitNs = 50000000ull;     // 50 ms per block
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, uint64_t deadline)
{
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() > deadline) return;
}

// ---- inter-block barriers inside one launch ------------------------------------------
// A group of blocks that are resident together (a grid sized to the resident
// capacity) meets at a barrier made of two words on their own 128-byte line:
// an arrival count that wraps to zero at the group size, and a generation
// that the last arrival advances.  Thread 0 of each block reads the
// generation once before its first arrival (it cannot advance before that
// arrival) and counts it up itself after every barrier, so a barrier costs
// one atomic and the polls; the same words serve any number of barriers in a
// row, for any group size, and are left as they were found (count 0).
__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// old = *p; *p = old >= wrap ? 0 : old + 1, acquire-release at GPU scope.
__device__ __forceinline__ uint32_t atom_inc_acq_rel_gpu(uint32_t *p, uint32_t wrap)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(wrap) : "memory");
    return old;
}

// The generation a block expects at its next barrier on `bar` (thread 0).
__device__ __forceinline__ uint32_t barrier_generation(const uint32_t *bar) { return ld_relaxed_gpu(bar + 1); }

// Every thread of the block calls it; thread 0 arrives for the block with
// `gen` the barrier's current generation (barrier_generation, then this
// call's own count).  The memory operations the block made before the call
// are visible to every block of the group after it: the block barrier makes
// them visible to thread 0, whose acquire-release arrival publishes them and
// acquires the others'.  Returns false if the wait ran out (MOIRA_DEV_TIMEOUT).
__device__ __forceinline__ bool group_barrier(uint32_t *bar, uint32_t n_blocks, uint32_t &gen, const WaitGuard &g,
                                              uint64_t limit_ns = kWaitLimitNs)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t old = atom_inc_acq_rel_gpu(bar, n_blocks - 1u);
        if (old == n_blocks - 1u) {
            st_release_gpu(bar + 1, gen + 1u);
        } else if (!guard_failed(g)) {
            const uint64_t t0 = globaltimer();
            while (ld_acquire_gpu(bar + 1) == gen) {
                if (guard_failed(g)) break;
                if (globaltimer() - t0 > limit_ns) {
                    guard_fail(g);
                    break;
                }
            }
        }
        gen += 1u;
    }
    __syncthreads();
    return !guard_failed(g);
}

// ---- shared-memory histograms ------------------------------------------------------
// hist[bin] += v for the active lanes.  When all active lanes of the warp hit
// the same bin (a flat mass distribution sends whole warps to one bin) their
// sum is added once; otherwise every lane adds its own.  Every lane of the
// warp must call it.
__device__ __forceinline__ void hist_add_warp(uint32_t *hist, uint32_t bin, uint32_t v, bool active)
{
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    int same;
    __match_all_sync(act, bin, &same);
    if (same) {
        const uint32_t sum = __reduce_add_sync(act, v);
        if (static_cast<int>(__ffs(act)) - 1 == static_cast<int>(threadIdx.x & 31)) atomicAdd(&hist[bin], sum);
    } else {
        atomicAdd(&hist[bin], v);
    }
}

// ---- programmatic dependent launch -------------------------------------------------
// A kernel launched with programmatic stream serialisation may start while its
// predecessor in the stream is still running.  pdl_wait() blocks until the
// predecessor grid has completed and its memory is visible; everything that
// reads or writes data shared with earlier kernels must come after it.
// pdl_trigger() lets the successor's blocks be scheduled early.  Both are
// no-ops for a normal launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- TMA ---------------------------------------------------------------------------
// 2-D tiled tensor load into this CTA's shared memory, completion counted in
// bytes on `bar`.  c0 is the inner (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t c0,
                                            int32_t c1, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// tma_load_2d with an L2 cache policy.
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int32_t c0,
                                                 int32_t c1, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

// 1-D bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
// from global memory into this CTA's shared memory, counted on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// L2 policy for data read once per step (the page summaries): its lines are
// evicted first.
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

// bulk_load with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                               uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- ldmatrix / mma ----------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D[16x8] += A[16x16] (row) * B[16x8] (col), bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same MMA with fp16 operands (fp32 accumulate).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace moira
