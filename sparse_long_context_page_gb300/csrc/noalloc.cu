// moira_select_noalloc: the coverage selection without a caller workspace.
//
// Some callers cannot allocate device memory at all: plug-ins that are
// handed only their input and output buffers, runtimes whose device memory
// is owned by another allocator, or a decode loop that must never call
// cudaMalloc (it synchronises the device and is not allowed in every stream
// capture mode).  moira_select needs scratch for the page weights and the
// per-chunk softmax normalisers; this entry point keeps that scratch in a
// fixed array compiled into the library instead, so it allocates nothing.
//
// The array is a file-scope static __device__ object of kNoAllocBytes: every
// GPU that loads the library holds it until the process exits.  Its device
// address is looked up once per device (cudaGetSymbolAddress) on the first
// call made with that device current, so that first call must not happen
// while a stream is being captured.  All calls share the array and it keeps
// the last call's contents; the kernels overwrite every scratch element they
// read, and the status word is cleared on every call.  Two calls that overlap
// on the GPU (different streams, or one call in flight while another starts)
// race on the array; calls issued in order on one stream do not.  The
// arguments are checked exactly as moira_select checks them (checks.h), and
// the stream must belong to the current device.
#include <cmath>
#include <mutex>

#include "../../include/moira.h"
#include "checks.h"
#include "moira_device.cuh"
#include "moira_launch.h"

constexpr size_t kNoAllocBytes = 4u << 20;      // MOIRA_NOALLOC_SCRATCH_BYTES
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

moira_status scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOIRA_ECUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOIRA_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return MOIRA_ECUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOIRA_OK;
}

}  // namespace

extern "C" moira_status moira_select_noalloc(const moira_shape *shape, const void *q,
                                             const void *summ, const int32_t *page_table,
                                             const int32_t *seq_lens, int32_t batch,
                                             int32_t max_pages, float gamma, float sm_scale,
                                             int32_t *lists, int32_t *lengths,
                                             moira_stream_t stream)
{
    using namespace moira;
    moira_status st = check_select_args(shape, MOIRA_SUMM_BF16, q, summ, page_table, seq_lens, batch,
                                        max_pages, MOIRA_RULE_COVERAGE, gamma, sm_scale, lists, lengths);
    if (st != MOIRA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the scratch address and the launches are the current device's: a
    // stream of another device is refused rather than launched into
    int cur = 0, sdev = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess)
        return MOIRA_ECUDA;
    if (sdev != cur) return MOIRA_EINVAL;

    // scratch: status word | page weights [batch][Hq][ld] | chunk (max, sum) [batch][Hq][ldc]
    const int hq = shape->num_q_heads;
    const size_t off_scores = 256;
    const size_t off_chunks =
        align_up(off_scores + sizeof(float) * static_cast<size_t>(batch) * hq * weights_ld(max_pages), 256);
    const size_t need = off_chunks + sizeof(float) * static_cast<size_t>(batch) * hq * chunks_ld(max_pages);
    if (need > kNoAllocBytes) return MOIRA_EUNSUPPORTED;     // beyond the compiled-in scratch

    void *base = nullptr;
    if ((st = scratch_address(&base)) != MOIRA_OK) return st;
    uint8_t *w = static_cast<uint8_t *>(base);
    uint32_t *status = reinterpret_cast<uint32_t *>(w);
    float *scores = reinterpret_cast<float *>(w + off_scores);
    float *chunks = reinterpret_cast<float *>(w + off_chunks);

    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return MOIRA_ECUDA;
    const bool dense = gamma >= 1.0f;
    const unsigned long long gfx =
        dense ? 0ull : static_cast<unsigned long long>(std::ceil(static_cast<double>(gamma) * 0x1p31));
    if (!dense) {
        const float scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
        if (launch_score(q, summ, kSummBf16, page_table, seq_lens, batch, hq, shape->num_kv_heads,
                         max_pages, shape->num_phys_pages, scale_log2, scores, chunks, false,
                         status, s) != cudaSuccess)
            return MOIRA_ECUDA;
    }
    if (launch_select(scores, chunks, page_table, seq_lens, batch, hq, shape->num_kv_heads,
                      max_pages, shape->num_phys_pages, kRuleCoverage, gfx, 0.f, dense, lists,
                      lengths, status, s) !=
        cudaSuccess)
        return MOIRA_ECUDA;
    return MOIRA_OK;
}
