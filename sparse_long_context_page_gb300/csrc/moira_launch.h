// Internal launch interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace moira {

// `fmt` is a summary format (kSummBf16 / kSummQ8 / kSummQ2, moira_device.cuh).
cudaError_t launch_summarize(const void *k_pool, void *summ, const int32_t *phys_pages, int n,
                             int hkv, long long num_pages, int fmt, uint32_t *status,
                             cudaStream_t stream);

cudaError_t launch_append(const void *k_new, const void *v_new, void *k_pool, void *v_pool,
                          void *summ, const int32_t *page_table, const int32_t *seq_lens,
                          int batch, int hkv, int max_pages, long long num_pages, int fmt,
                          cudaStream_t stream);

// `early`: the launch directly follows a kernel of this library that writes
// neither page_table nor seq_lens (the previous layer's attention inside one
// decode step); the kernel then reads them before its dependency wait.
cudaError_t launch_score(const void *q, const void *summ, int fmt, const int32_t *page_table,
                         const int32_t *seq_lens, int batch, int hq, int hkv, int max_pages,
                         long long num_pages, float scale_log2, float *scores, float *chunks,
                         bool early, uint32_t *status, cudaStream_t stream);

// Page rules of the selection (the values of the public moira_rule).
constexpr int kRuleCoverage = 0;          // target = ceil(gamma * 2^31)
constexpr int kRuleTopK = 1;              // target = k pages
constexpr int kRuleTopDelta = 2;          // delta: keep mass >= delta * max mass

cudaError_t launch_select(const float *scores, const float *chunks, const int32_t *page_table,
                          const int32_t *seq_lens, int batch, int hq, int hkv, int max_pages,
                          long long num_pages, int rule, unsigned long long target, float delta,
                          bool dense, int32_t *lists, int32_t *lengths, uint32_t *status,
                          cudaStream_t stream);

struct AttendArgs {
    const void *q;
    const int32_t *lists;
    const int32_t *lengths;
    const int32_t *seq_lens;
    float *out;
    float *partials;
    uint32_t *counters;
    uint32_t *gcounters;
    uint32_t *status;
    int hq, hkv, units, max_pages;
    long long num_pages;
    float scale_log2;
#ifdef MOIRA_CTA_TIMES
    unsigned long long *cta_times;   // [grid][2] (start, end) %globaltimer per block, or null
#endif
};

#ifdef MOIRA_CTA_TIMES
// Where the next attention launch records its per-block times (null: none);
// advanced by one grid's worth per launch, up to the set number of launches.
unsigned long long *next_cta_times(int blocks);
#endif

cudaError_t launch_attend(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                          const AttendArgs &args, int blocks, cudaStream_t stream);

// The selection and the attention of one layer in one launch (k_select_attend,
// fused.cu), for small batches: every list's selection is spread over the
// grid's blocks, which meet at barriers inside the launch, then the same
// blocks attend.  `at.lists` is unused (the kept pages come from the
// selection); the outputs lists / lengths are written as moira_select would.
// With `dense` every page is kept and no estimate runs (no k_score before it).
struct FusedArgs {
    AttendArgs at;                 // at.lists / at.lengths: the outputs, read back by the attention
    const float *weights;          // k_score's chunk-relative weights
    const float *chunks;           // k_score's per-chunk (max, sum)
    const int32_t *page_table;
    int32_t *lists;                // out
    int32_t *lengths;              // out
    uint32_t *bars;                // [kFusedMaxUnits + 1][kBarWords]
    uint32_t *l1hist;              // [units][kL1Stride]
    uint32_t *mass;                // [units][ld]
    unsigned long long target;     // gamma on the 2^-31 grid
    int ld, ldc;
    int dense;
};

// Whether k_select_attend takes `units` lists of at most `max_pages` pages on
// a grid of `blocks` (and fits 2 blocks per SM on the current device).
bool select_attend_fits(int units, int max_pages, int blocks);

// The coverage selection in one launch, one thread-block cluster per list
// (k_cover, cover.cu): the cluster size a launch of `units` lists takes (16
// or 8), or 0 when the device cannot hold every list's cluster at once or
// max_pages needs more than two rounds of chunks per block; then the launch
// itself (bf16 summaries; target = gamma on the 2^-31 grid, rounded up).
int cover_cluster_size(int units, int max_pages);
cudaError_t launch_cover(const void *q, const void *summ, const int32_t *page_table, const int32_t *seq_lens,
                         int batch, int hq, int hkv, int max_pages, long long num_pages, float scale_log2,
                         unsigned long long target, bool early, int32_t *lists, int32_t *lengths,
                         uint32_t *status, int C, cudaStream_t stream);
cudaError_t launch_select_attend(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                 const FusedArgs &args, int blocks, cudaStream_t stream);

int attend_blocks_per_sm();

// Diagnostics of bounded waits made to run out (see diag.cu).
cudaError_t launch_wait_timeout(uint32_t *status, unsigned long long limit_ns, cudaStream_t stream);
cudaError_t launch_wait_chain(uint32_t *status, unsigned long long limit_ns, int n_waits, cudaStream_t stream);
cudaError_t launch_barrier_timeout(uint32_t *status, uint32_t *bar, int blocks, unsigned long long limit_ns,
                                   cudaStream_t stream);

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute stays set in the device's context, so it is
// set once per (kernel, device, larger size) instead of on every launch; the
// caller keeps the per-device record (`seen`, 64 devices).
template <typename Kernel>
cudaError_t raise_smem_limit(Kernel kernel, size_t bytes, std::atomic<int> *seen)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(bytes));
    if (seen[dev].load(std::memory_order_relaxed) >= static_cast<int>(bytes)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(bytes));
    if (e == cudaSuccess) seen[dev].store(static_cast<int>(bytes), std::memory_order_relaxed);
    return e;
}

// Launch with programmatic stream serialisation (see pdl_wait / pdl_trigger).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace moira
