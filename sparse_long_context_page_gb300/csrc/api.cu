// C ABI of the sparse-decode library: host-side argument checks, workspace
// carving, TMA descriptor encoding and kernel launches.  Nothing here
// allocates, synchronises or reads device memory inside select/attend/step.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/moira.h"
#ifdef MOIRA_CTA_TIMES
#include "../../include/moira_cta_times.h"
#endif
#include "checks.h"
#include "moira_device.cuh"
#include "moira_launch.h"

using namespace moira;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

// The attention grid: every SM holds attend_blocks_per_sm() resident blocks
// (one wave; each block takes an equal range of the concatenated lists).
int attend_blocks() { return current_sm_count() * attend_blocks_per_sm(); }

WsLayout layout_for(const moira_shape *s, int32_t batch, int32_t max_pages)
{
    return ws_layout(batch, s->num_q_heads, max_pages, batch * s->num_kv_heads, attend_blocks());
}

moira_status check_ws(const moira_shape *s, int32_t batch, int32_t max_pages, void *ws, size_t bytes)
{
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOIRA_EWORKSPACE;
    if (bytes < layout_for(s, batch, max_pages).total) return MOIRA_EWORKSPACE;
    return MOIRA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// One layer's pool viewed as a 2-D bf16 tensor [P * Hkv * S rows][d], loaded
// in boxes of 16 rows x 64 elements (128 bytes) with the 128-byte swizzle.
bool make_pool_map(CUtensorMap *map, const void *pool, const moira_shape *s)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim),
                          static_cast<cuuint64_t>(s->num_phys_pages) * s->num_kv_heads * kPageSize};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kPageSize)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(pool), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

moira_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOIRA_OK : MOIRA_ECUDA; }

moira_status select_impl(const moira_shape *shape, int32_t fmt, const void *q, const void *summ,
                         const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                         int32_t max_pages, int32_t rule, float param, float sm_scale,
                         int32_t *lists, int32_t *lengths, void *ws, size_t ws_bytes,
                         bool early, cudaStream_t stream)
{
    static_assert(MOIRA_RULE_COVERAGE == kRuleCoverage && MOIRA_RULE_TOPK == kRuleTopK &&
                      MOIRA_RULE_TOPDELTA == kRuleTopDelta,
                  "public rule values match the kernels'");
    static_assert(MOIRA_SUMM_BF16 == kSummBf16 && MOIRA_SUMM_Q8 == kSummQ8 && MOIRA_SUMM_Q2 == kSummQ2,
                  "public summary formats match the kernels'");
    const float gamma = rule == MOIRA_RULE_COVERAGE ? param : 0.5f;
    const WsLayout L = layout_for(shape, batch, max_pages);
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *status = reinterpret_cast<uint32_t *>(w + L.status);
    float *scores = reinterpret_cast<float *>(w + L.scores);
    float *chunks = reinterpret_cast<float *>(w + L.chunks);
    const bool dense = rule == MOIRA_RULE_COVERAGE && gamma >= 1.0f;
    // coverage: gamma on the 2^-31 fixed-point grid of the mass histograms,
    // rounded up; top-k: the page count
    unsigned long long gfx = 0ull;
    if (rule == MOIRA_RULE_COVERAGE && !dense)
        gfx = static_cast<unsigned long long>(std::ceil(static_cast<double>(gamma) * 0x1p31));
    else if (rule == MOIRA_RULE_TOPK)
        gfx = static_cast<unsigned long long>(param);
    const float delta = rule == MOIRA_RULE_TOPDELTA ? param : 0.f;
    if (!dense) {
        const float scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
        cudaError_t e = launch_score(q, summ, fmt, page_table, seq_lens, batch, shape->num_q_heads,
                                     shape->num_kv_heads, max_pages, shape->num_phys_pages,
                                     scale_log2, scores, chunks, early, status, stream);
        if (e != cudaSuccess) return MOIRA_ECUDA;
    }
    return cuda_status(launch_select(scores, chunks, page_table, seq_lens, batch,
                                     shape->num_q_heads, shape->num_kv_heads, max_pages,
                                     shape->num_phys_pages, rule, gfx, delta, dense, lists,
                                     lengths, status, stream));
}

moira_status attend_impl(const moira_shape *shape, const void *q, const void *k_pool,
                         const void *v_pool, const int32_t *lists, const int32_t *lengths,
                         const int32_t *seq_lens, int32_t batch, int32_t max_pages, float sm_scale,
                         float *out, void *ws, size_t ws_bytes, cudaStream_t stream)
{
    const WsLayout L = layout_for(shape, batch, max_pages);
    uint8_t *w = static_cast<uint8_t *>(ws);
    CUtensorMap mk, mv;
    if (!make_pool_map(&mk, k_pool, shape) || !make_pool_map(&mv, v_pool, shape)) return MOIRA_ECUDA;
    AttendArgs a;
    a.q = q;
    a.lists = lists;
    a.lengths = lengths;
    a.seq_lens = seq_lens;
    a.out = out;
    a.partials = reinterpret_cast<float *>(w + L.partials);
    a.counters = reinterpret_cast<uint32_t *>(w + L.counters);
    a.gcounters = reinterpret_cast<uint32_t *>(w + L.gcounters);
    a.status = reinterpret_cast<uint32_t *>(w + L.status);
    a.hq = shape->num_q_heads;
    a.hkv = shape->num_kv_heads;
    a.units = batch * shape->num_kv_heads;
    a.max_pages = max_pages;
    a.num_pages = shape->num_phys_pages;
    a.scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
#ifdef MOIRA_CTA_TIMES
    a.cta_times = next_cta_times(attend_blocks());
#endif
    return cuda_status(launch_attend(mk, mv, a, attend_blocks(), stream));
}

// One layer's selection and attention.  Small batches (fewer than 64 lists
// of at most 16 chunks per selecting block) with the coverage rule run as
// k_score then one k_select_attend launch; everything else as select_impl
// then attend_impl.  Both give the same lists and lengths bit for bit.
moira_status select_attend_impl(const moira_shape *shape, int32_t fmt, const void *q, const void *summ,
                                const void *k_pool, const void *v_pool, const int32_t *page_table,
                                const int32_t *seq_lens, int32_t batch, int32_t max_pages, int32_t rule,
                                float param, float sm_scale, int32_t *lists, int32_t *lengths, float *out,
                                void *ws, size_t ws_bytes, bool early, cudaStream_t stream)
{
    const int units = batch * shape->num_kv_heads;
    const int blocks = attend_blocks();
    if (rule != MOIRA_RULE_COVERAGE || !select_attend_fits(units, max_pages, blocks)) {
        moira_status st = select_impl(shape, fmt, q, summ, page_table, seq_lens, batch, max_pages, rule, param,
                                      sm_scale, lists, lengths, ws, ws_bytes, early, stream);
        if (st != MOIRA_OK) return st;
        return attend_impl(shape, q, k_pool, v_pool, lists, lengths, seq_lens, batch, max_pages, sm_scale, out,
                           ws, ws_bytes, stream);
    }
    const WsLayout L = layout_for(shape, batch, max_pages);
    uint8_t *w = static_cast<uint8_t *>(ws);
    const float gamma = param;
    const bool dense = gamma >= 1.0f;
    const float scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
    uint32_t *status = reinterpret_cast<uint32_t *>(w + L.status);
    float *scores = reinterpret_cast<float *>(w + L.scores);
    float *chunks = reinterpret_cast<float *>(w + L.chunks);
    if (!dense) {
        cudaError_t e = launch_score(q, summ, fmt, page_table, seq_lens, batch, shape->num_q_heads,
                                     shape->num_kv_heads, max_pages, shape->num_phys_pages, scale_log2, scores,
                                     chunks, early, status, stream);
        if (e != cudaSuccess) return MOIRA_ECUDA;
    }
    CUtensorMap mk, mv;
    if (!make_pool_map(&mk, k_pool, shape) || !make_pool_map(&mv, v_pool, shape)) return MOIRA_ECUDA;
    FusedArgs f;
    f.at.q = q;
    f.at.lists = lists;
    f.at.lengths = lengths;
    f.at.seq_lens = seq_lens;
    f.at.out = out;
    f.at.partials = reinterpret_cast<float *>(w + L.partials);
    f.at.counters = reinterpret_cast<uint32_t *>(w + L.counters);
    f.at.gcounters = reinterpret_cast<uint32_t *>(w + L.gcounters);
    f.at.status = status;
    f.at.hq = shape->num_q_heads;
    f.at.hkv = shape->num_kv_heads;
    f.at.units = units;
    f.at.max_pages = max_pages;
    f.at.num_pages = shape->num_phys_pages;
    f.at.scale_log2 = scale_log2;
#ifdef MOIRA_CTA_TIMES
    f.at.cta_times = next_cta_times(blocks);
#endif
    f.weights = scores;
    f.chunks = chunks;
    f.page_table = page_table;
    f.lists = lists;
    f.lengths = lengths;
    f.bars = reinterpret_cast<uint32_t *>(w + L.fbars);
    f.l1hist = reinterpret_cast<uint32_t *>(w + L.fl1);
    f.mass = reinterpret_cast<uint32_t *>(w + L.fmass);
    f.target = dense ? 0ull : static_cast<unsigned long long>(std::ceil(static_cast<double>(gamma) * 0x1p31));
    f.ld = weights_ld(max_pages);
    f.ldc = chunks_ld(max_pages);
    f.dense = dense ? 1 : 0;
    return cuda_status(launch_select_attend(mk, mv, f, blocks, stream));
}

}  // namespace

// ---------------------------------------------------------------- argument checks (checks.h)

namespace {

bool finite_pos(float x) { return std::isfinite(x) && x > 0.f; }

bool valid_format(int32_t fmt)
{
    return fmt == MOIRA_SUMM_BF16 || fmt == MOIRA_SUMM_Q8 || fmt == MOIRA_SUMM_Q2;
}

// The range of each rule's parameter (moira_rule).
bool valid_rule(int32_t rule, float param)
{
    switch (rule) {
    case MOIRA_RULE_COVERAGE:
    case MOIRA_RULE_TOPDELTA:
        return param > 0.f && param <= 1.f;
    case MOIRA_RULE_TOPK:
        return param >= 0.f && param <= 16777216.f && param == std::floor(param);
    default:
        return false;
    }
}

bool aligned16_ptr(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace moira {

moira_status check_shape(const moira_shape *s)
{
    if (!s) return MOIRA_EINVAL;
    if (s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->head_dim <= 0 || s->page_size <= 0 ||
        s->num_phys_pages <= 0)
        return MOIRA_EINVAL;
    if (s->num_q_heads % s->num_kv_heads != 0) return MOIRA_EINVAL;
    if (s->head_dim != kHeadDim || s->page_size != kPageSize) return MOIRA_EUNSUPPORTED;
    if (s->num_q_heads / s->num_kv_heads != kGroup) return MOIRA_EUNSUPPORTED;
    if (32 % s->num_kv_heads != 0) return MOIRA_EUNSUPPORTED;       // Hkv in {1, 2, 4, 8}
    // TMA row coordinates are 32-bit: P * Hkv * S rows per layer pool.
    if (s->num_phys_pages * s->num_kv_heads * kPageSize >= (1LL << 31)) return MOIRA_EUNSUPPORTED;
    return MOIRA_OK;
}

moira_status check_batch(const moira_shape *s, int32_t batch, int32_t max_pages)
{
    if (batch <= 0 || max_pages <= 0) return MOIRA_EINVAL;
    if (max_pages > kMaxPagesPerSeq) return MOIRA_EUNSUPPORTED;
    if (static_cast<long long>(batch) * s->num_kv_heads > kMaxUnits) return MOIRA_EUNSUPPORTED;
    return MOIRA_OK;
}

moira_status check_select_args(const moira_shape *shape, int32_t fmt, const void *q, const void *summ,
                               const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                               int32_t max_pages, int32_t rule, float param, float sm_scale,
                               const int32_t *lists, const int32_t *lengths)
{
    moira_status st = check_shape(shape);
    if (st != MOIRA_OK) return st;
    if ((st = check_batch(shape, batch, max_pages)) != MOIRA_OK) return st;
    if (!valid_format(fmt) || !valid_rule(rule, param) || !finite_pos(sm_scale)) return MOIRA_EINVAL;
    if (!q || !summ || !page_table || !seq_lens || !lists || !lengths) return MOIRA_EINVAL;
    if (!aligned16_ptr(q) || !aligned16_ptr(summ)) return MOIRA_EINVAL;
    return MOIRA_OK;
}

}  // namespace moira

#ifdef MOIRA_CTA_TIMES
// Load-balance build only (include/moira_cta_times.h): where the next
// attention launches record their per-block times.
static unsigned long long *g_cta_times = nullptr;
static int g_cta_launches = 0;

unsigned long long *moira::next_cta_times(int blocks)
{
    if (g_cta_times == nullptr || g_cta_launches <= 0) return nullptr;
    unsigned long long *p = g_cta_times;
    g_cta_times += 2 * static_cast<size_t>(blocks);
    if (--g_cta_launches == 0) g_cta_times = nullptr;
    return p;
}
#endif

extern "C" {

size_t moira_workspace_bytes(const moira_shape *shape, int32_t batch, int32_t max_pages)
{
    if (check_shape(shape) != MOIRA_OK || check_batch(shape, batch, max_pages) != MOIRA_OK) return 0;
    if (attend_blocks() <= 0) return 0;
    return layout_for(shape, batch, max_pages).total;
}

moira_status moira_workspace_init(void *workspace, size_t ws_bytes, moira_stream_t stream)
{
    if (!workspace || ws_bytes == 0) return MOIRA_EWORKSPACE;
    return cuda_status(cudaMemsetAsync(workspace, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moira_summary_page_bytes(const moira_shape *shape, int32_t format)
{
    if (check_shape(shape) != MOIRA_OK || !valid_format(format)) return 0;
    return static_cast<size_t>(summ_page_bytes(format, shape->num_kv_heads));
}

moira_status moira_update_summaries_ex(const moira_shape *shape, int32_t format, const void *k_pool,
                                       void *summ, const int32_t *phys_pages, int32_t n,
                                       moira_stream_t stream)
{
    moira_status st = check_shape(shape);
    if (st != MOIRA_OK) return st;
    if (!valid_format(format)) return MOIRA_EINVAL;
    if (n < 0 || (n > 0 && (!k_pool || !summ || !phys_pages))) return MOIRA_EINVAL;
    if (n == 0) return MOIRA_OK;
    if (!aligned16(k_pool) || !aligned16(summ)) return MOIRA_EINVAL;
    // This call takes no workspace, so there is no status word: page ids out
    // of range are skipped without a record (select and attend flag them).
    return cuda_status(launch_summarize(k_pool, summ, phys_pages, n, shape->num_kv_heads,
                                        shape->num_phys_pages, format, nullptr,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

moira_status moira_update_summaries(const moira_shape *shape, const void *k_pool, void *summ,
                                    const int32_t *phys_pages, int32_t n, moira_stream_t stream)
{
    return moira_update_summaries_ex(shape, MOIRA_SUMM_BF16, k_pool, summ, phys_pages, n, stream);
}

moira_status moira_append_kv_ex(const moira_shape *shape, int32_t format, const void *k_new,
                                const void *v_new, void *k_pool, void *v_pool, void *summ,
                                const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                                int32_t max_pages, moira_stream_t stream)
{
    moira_status st = check_shape(shape);
    if (st != MOIRA_OK) return st;
    if ((st = check_batch(shape, batch, max_pages)) != MOIRA_OK) return st;
    if (!valid_format(format)) return MOIRA_EINVAL;
    if (!k_new || !v_new || !k_pool || !v_pool || !summ || !page_table || !seq_lens)
        return MOIRA_EINVAL;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
        !aligned16(summ))
        return MOIRA_EINVAL;
    return cuda_status(launch_append(k_new, v_new, k_pool, v_pool, summ, page_table, seq_lens,
                                     batch, shape->num_kv_heads, max_pages, shape->num_phys_pages,
                                     format, reinterpret_cast<cudaStream_t>(stream)));
}

moira_status moira_append_kv(const moira_shape *shape, const void *k_new, const void *v_new,
                             void *k_pool, void *v_pool, void *summ, const int32_t *page_table,
                             const int32_t *seq_lens, int32_t batch, int32_t max_pages,
                             moira_stream_t stream)
{
    return moira_append_kv_ex(shape, MOIRA_SUMM_BF16, k_new, v_new, k_pool, v_pool, summ,
                              page_table, seq_lens, batch, max_pages, stream);
}

moira_status moira_select_ex(const moira_shape *shape, int32_t format, const void *q,
                             const void *summ, const int32_t *page_table, const int32_t *seq_lens,
                             int32_t batch, int32_t max_pages, int32_t rule, float param,
                             float sm_scale, int32_t *lists, int32_t *lengths, void *workspace,
                             size_t ws_bytes, moira_stream_t stream)
{
    moira_status st = check_select_args(shape, format, q, summ, page_table, seq_lens, batch, max_pages,
                                        rule, param, sm_scale, lists, lengths);
    if (st != MOIRA_OK) return st;
    if ((st = check_ws(shape, batch, max_pages, workspace, ws_bytes)) != MOIRA_OK) return st;
    return select_impl(shape, format, q, summ, page_table, seq_lens, batch, max_pages, rule, param,
                       sm_scale, lists, lengths, workspace, ws_bytes, false,
                       reinterpret_cast<cudaStream_t>(stream));
}

moira_status moira_select(const moira_shape *shape, const void *q, const void *summ,
                          const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                          int32_t max_pages, float gamma, float sm_scale, int32_t *lists,
                          int32_t *lengths, void *workspace, size_t ws_bytes, moira_stream_t stream)
{
    return moira_select_ex(shape, MOIRA_SUMM_BF16, q, summ, page_table, seq_lens, batch, max_pages,
                           MOIRA_RULE_COVERAGE, gamma, sm_scale, lists, lengths, workspace,
                           ws_bytes, stream);
}

moira_status moira_select_rule(const moira_shape *shape, const void *q, const void *summ,
                               const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                               int32_t max_pages, int32_t rule, float param, float sm_scale,
                               int32_t *lists, int32_t *lengths, void *workspace, size_t ws_bytes,
                               moira_stream_t stream)
{
    return moira_select_ex(shape, MOIRA_SUMM_BF16, q, summ, page_table, seq_lens, batch, max_pages,
                           rule, param, sm_scale, lists, lengths, workspace, ws_bytes, stream);
}

moira_status moira_select_clustered(const moira_shape *shape, const void *q, const void *summ,
                                    const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                                    int32_t max_pages, float gamma, float sm_scale, int32_t *lists,
                                    int32_t *lengths, void *workspace, size_t ws_bytes, moira_stream_t stream)
{
    moira_status st = check_select_args(shape, MOIRA_SUMM_BF16, q, summ, page_table, seq_lens, batch, max_pages,
                                        MOIRA_RULE_COVERAGE, gamma, sm_scale, lists, lengths);
    if (st != MOIRA_OK) return st;
    if ((st = check_ws(shape, batch, max_pages, workspace, ws_bytes)) != MOIRA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (gamma >= 1.0f)                                   // dense: no estimate, as moira_select
        return select_impl(shape, MOIRA_SUMM_BF16, q, summ, page_table, seq_lens, batch, max_pages,
                           MOIRA_RULE_COVERAGE, gamma, sm_scale, lists, lengths, workspace, ws_bytes, false, s);
    const int C = cover_cluster_size(batch * shape->num_kv_heads, max_pages);
    if (C == 0) return MOIRA_EUNSUPPORTED;
    const WsLayout L = layout_for(shape, batch, max_pages);
    uint32_t *status = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(workspace) + L.status);
    const float scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
    const unsigned long long gfx = static_cast<unsigned long long>(std::ceil(static_cast<double>(gamma) * 0x1p31));
    return cuda_status(launch_cover(q, summ, page_table, seq_lens, batch, shape->num_q_heads, shape->num_kv_heads,
                                    max_pages, shape->num_phys_pages, scale_log2, gfx, false, lists, lengths,
                                    status, C, s));
}

int32_t moira_select_cluster_size(const moira_shape *shape, int32_t batch, int32_t max_pages)
{
    if (check_shape(shape) != MOIRA_OK || check_batch(shape, batch, max_pages) != MOIRA_OK) return 0;
    return cover_cluster_size(batch * shape->num_kv_heads, max_pages);
}

moira_status moira_attend(const moira_shape *shape, const void *q, const void *k_pool,
                          const void *v_pool, const int32_t *lists, const int32_t *lengths,
                          const int32_t *seq_lens, int32_t batch, int32_t max_pages,
                          float sm_scale, float *out, void *workspace, size_t ws_bytes,
                          moira_stream_t stream)
{
    moira_status st = check_shape(shape);
    if (st != MOIRA_OK) return st;
    if ((st = check_batch(shape, batch, max_pages)) != MOIRA_OK) return st;
    if (!finite_pos(sm_scale)) return MOIRA_EINVAL;
    if (!q || !k_pool || !v_pool || !lists || !lengths || !seq_lens || !out) return MOIRA_EINVAL;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return MOIRA_EINVAL;
    if ((st = check_ws(shape, batch, max_pages, workspace, ws_bytes)) != MOIRA_OK) return st;
    return attend_impl(shape, q, k_pool, v_pool, lists, lengths, seq_lens, batch, max_pages,
                       sm_scale, out, workspace, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

moira_status moira_select_attend_ex(const moira_shape *shape, int32_t format, const void *q,
                                    const void *summ, const void *k_pool, const void *v_pool,
                                    const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                                    int32_t max_pages, float gamma, float sm_scale, int32_t *lists,
                                    int32_t *lengths, float *out, void *workspace, size_t ws_bytes,
                                    moira_stream_t stream)
{
    moira_status st = check_shape(shape);
    if (st != MOIRA_OK) return st;
    if ((st = check_batch(shape, batch, max_pages)) != MOIRA_OK) return st;
    if (!valid_format(format) || !valid_rule(MOIRA_RULE_COVERAGE, gamma) || !finite_pos(sm_scale))
        return MOIRA_EINVAL;
    if (!q || !summ || !k_pool || !v_pool || !page_table || !seq_lens || !lists || !lengths || !out)
        return MOIRA_EINVAL;
    if (!aligned16(q) || !aligned16(summ) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
        return MOIRA_EINVAL;
    if ((st = check_ws(shape, batch, max_pages, workspace, ws_bytes)) != MOIRA_OK) return st;
    return select_attend_impl(shape, format, q, summ, k_pool, v_pool, page_table, seq_lens, batch, max_pages,
                              MOIRA_RULE_COVERAGE, gamma, sm_scale, lists, lengths, out, workspace, ws_bytes,
                              false, reinterpret_cast<cudaStream_t>(stream));
}

moira_status moira_select_attend(const moira_shape *shape, const void *q, const void *summ,
                                 const void *k_pool, const void *v_pool, const int32_t *page_table,
                                 const int32_t *seq_lens, int32_t batch, int32_t max_pages, float gamma,
                                 float sm_scale, int32_t *lists, int32_t *lengths, float *out,
                                 void *workspace, size_t ws_bytes, moira_stream_t stream)
{
    return moira_select_attend_ex(shape, MOIRA_SUMM_BF16, q, summ, k_pool, v_pool, page_table, seq_lens,
                                  batch, max_pages, gamma, sm_scale, lists, lengths, out, workspace, ws_bytes,
                                  stream);
}

moira_status moira_score_ex(const moira_shape *shape, int32_t format, const void *q, const void *summ,
                            const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                            int32_t max_pages, float sm_scale, void *workspace, size_t ws_bytes,
                            moira_stream_t stream)
{
    moira_status st = check_shape(shape);
    if (st != MOIRA_OK) return st;
    if ((st = check_batch(shape, batch, max_pages)) != MOIRA_OK) return st;
    if (!valid_format(format) || !finite_pos(sm_scale)) return MOIRA_EINVAL;
    if (!q || !summ || !page_table || !seq_lens) return MOIRA_EINVAL;
    if (!aligned16(q) || !aligned16(summ)) return MOIRA_EINVAL;
    if ((st = check_ws(shape, batch, max_pages, workspace, ws_bytes)) != MOIRA_OK) return st;
    const WsLayout L = layout_for(shape, batch, max_pages);
    uint8_t *w = static_cast<uint8_t *>(workspace);
    const float scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634);
    return cuda_status(launch_score(q, summ, format, page_table, seq_lens, batch, shape->num_q_heads,
                                    shape->num_kv_heads, max_pages, shape->num_phys_pages, scale_log2,
                                    reinterpret_cast<float *>(w + L.scores), reinterpret_cast<float *>(w + L.chunks),
                                    false, reinterpret_cast<uint32_t *>(w + L.status),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int32_t moira_select_attend_is_fused(const moira_shape *shape, int32_t batch, int32_t max_pages)
{
    if (check_shape(shape) != MOIRA_OK || check_batch(shape, batch, max_pages) != MOIRA_OK) return 0;
    return select_attend_fits(batch * shape->num_kv_heads, max_pages, attend_blocks()) ? 1 : 0;
}

moira_status moira_decode_step_ex(const moira_shape *shape, int32_t format, int32_t num_layers,
                                  const void *q_all, const void *k_pool_all,
                                  const void *v_pool_all, const void *summ_all,
                                  const int32_t *page_table, const int32_t *seq_lens,
                                  int32_t batch, int32_t max_pages, int32_t rule, float param,
                                  float sm_scale, int32_t *lists, int32_t *lengths_all,
                                  float *out_all, void *workspace, size_t ws_bytes,
                                  moira_stream_t stream)
{
    moira_status st = check_shape(shape);
    if (st != MOIRA_OK) return st;
    if ((st = check_batch(shape, batch, max_pages)) != MOIRA_OK) return st;
    if (num_layers <= 0) return MOIRA_EINVAL;
    if (!valid_format(format) || !valid_rule(rule, param) || !finite_pos(sm_scale))
        return MOIRA_EINVAL;
    if (!q_all || !k_pool_all || !v_pool_all || !summ_all || !page_table || !seq_lens || !lists ||
        !lengths_all || !out_all)
        return MOIRA_EINVAL;
    if (!aligned16(q_all) || !aligned16(k_pool_all) || !aligned16(v_pool_all) ||
        !aligned16(summ_all) || !aligned16(out_all))
        return MOIRA_EINVAL;
    if ((st = check_ws(shape, batch, max_pages, workspace, ws_bytes)) != MOIRA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t d = kHeadDim;
    const size_t q_layer = static_cast<size_t>(batch) * shape->num_q_heads * d;      // elements
    const size_t kv_layer = static_cast<size_t>(shape->num_phys_pages) * shape->num_kv_heads * kPageSize * d;
    const size_t sm_layer = static_cast<size_t>(shape->num_phys_pages) *
                            summ_page_bytes(format, shape->num_kv_heads);            // bytes
    const size_t len_layer = static_cast<size_t>(batch) * shape->num_kv_heads;
    const uint16_t *q = static_cast<const uint16_t *>(q_all);
    const uint16_t *kp = static_cast<const uint16_t *>(k_pool_all);
    const uint16_t *vp = static_cast<const uint16_t *>(v_pool_all);
    const uint8_t *sp = static_cast<const uint8_t *>(summ_all);
    for (int l = 0; l < num_layers; ++l) {
        st = select_impl(shape, format, q + l * q_layer, sp + l * sm_layer, page_table, seq_lens,
                         batch, max_pages, rule, param, sm_scale, lists,
                         lengths_all + l * len_layer, workspace, ws_bytes, l > 0, s);
        if (st != MOIRA_OK) return st;
        st = attend_impl(shape, q + l * q_layer, kp + l * kv_layer, vp + l * kv_layer, lists,
                         lengths_all + l * len_layer, seq_lens, batch, max_pages, sm_scale,
                         out_all + l * q_layer, workspace, ws_bytes, s);
        if (st != MOIRA_OK) return st;
    }
    return MOIRA_OK;
}

moira_status moira_decode_step(const moira_shape *shape, int32_t num_layers, const void *q_all,
                               const void *k_pool_all, const void *v_pool_all,
                               const void *summ_all, const int32_t *page_table,
                               const int32_t *seq_lens, int32_t batch, int32_t max_pages,
                               float gamma, float sm_scale, int32_t *lists, int32_t *lengths_all,
                               float *out_all, void *workspace, size_t ws_bytes,
                               moira_stream_t stream)
{
    return moira_decode_step_ex(shape, MOIRA_SUMM_BF16, num_layers, q_all, k_pool_all, v_pool_all,
                                summ_all, page_table, seq_lens, batch, max_pages,
                                MOIRA_RULE_COVERAGE, gamma, sm_scale, lists, lengths_all, out_all,
                                workspace, ws_bytes, stream);
}

moira_status moira_decode_step_host(const moira_shape *shape, int32_t num_layers,
                                    const void *q_host, void *q_dev, const void *k_pool_all,
                                    const void *v_pool_all, const void *summ_all,
                                    const int32_t *page_table, const int32_t *seq_lens,
                                    int32_t batch, int32_t max_pages, float gamma, float sm_scale,
                                    int32_t *lists, int32_t *lengths_all, float *out_dev,
                                    float *out_host, void *workspace, size_t ws_bytes,
                                    moira_stream_t stream)
{
    moira_status st = check_shape(shape);
    if (st != MOIRA_OK) return st;
    if ((st = check_batch(shape, batch, max_pages)) != MOIRA_OK) return st;
    if (num_layers <= 0 || !q_host || !out_host || !q_dev || !out_dev) return MOIRA_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t n = static_cast<size_t>(num_layers) * batch * shape->num_q_heads * kHeadDim;
    if (cudaMemcpyAsync(q_dev, q_host, n * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOIRA_ECUDA;
    st = moira_decode_step(shape, num_layers, q_dev, k_pool_all, v_pool_all, summ_all, page_table,
                           seq_lens, batch, max_pages, gamma, sm_scale, lists, lengths_all, out_dev,
                           workspace, ws_bytes, stream);
    if (st != MOIRA_OK) return st;
    return cuda_status(cudaMemcpyAsync(out_host, out_dev, n * 4, cudaMemcpyDeviceToHost, s));
}

moira_status moira_read_device_status(void *workspace, size_t ws_bytes, uint32_t *status_out,
                                      int32_t clear, moira_stream_t stream)
{
    if (!workspace || ws_bytes < 256) return MOIRA_EWORKSPACE;
    if (!status_out) return MOIRA_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOIRA_ECUDA;
    if (cudaMemcpy(status_out, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOIRA_ECUDA;
    if (clear) {
        if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return MOIRA_ECUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return MOIRA_ECUDA;
    }
    return MOIRA_OK;
}

int32_t moira_attend_grid_blocks(void) { return attend_blocks(); }

moira_status moira_diag_wait_timeout(void *workspace, size_t ws_bytes, uint64_t limit_ns,
                                     moira_stream_t stream)
{
    if (!workspace || ws_bytes < 256 || limit_ns < 1 || limit_ns > 10000000000ull) return MOIRA_EINVAL;
    return cuda_status(launch_wait_timeout(static_cast<uint32_t *>(workspace), limit_ns,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

moira_status moira_diag_wait_chain(void *workspace, size_t ws_bytes, uint64_t limit_ns, int32_t n_waits,
                                   moira_stream_t stream)
{
    if (!workspace || ws_bytes < 256 || limit_ns < 1 || limit_ns > 10000000000ull || n_waits < 1 ||
        n_waits > 4096)
        return MOIRA_EINVAL;
    return cuda_status(launch_wait_chain(static_cast<uint32_t *>(workspace), limit_ns, n_waits,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

moira_status moira_diag_barrier_timeout(void *workspace, size_t ws_bytes, uint64_t limit_ns, int32_t blocks,
                                        moira_stream_t stream)
{
    if (!workspace || ws_bytes < 256 || limit_ns < 1 || limit_ns > 10000000000ull || blocks < 1 ||
        blocks > current_sm_count())
        return MOIRA_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the barrier's two words sit on the status line's second 128 bytes,
    // cleared before the launch (the barrier never completes, so it leaves
    // its count behind) and after it
    uint32_t *bar = static_cast<uint32_t *>(workspace) + 32;
    if (cudaMemsetAsync(bar, 0, 128, s) != cudaSuccess) return MOIRA_ECUDA;
    if (launch_barrier_timeout(static_cast<uint32_t *>(workspace), bar, blocks, limit_ns, s) != cudaSuccess)
        return MOIRA_ECUDA;
    return cuda_status(cudaMemsetAsync(bar, 0, 128, s));
}

#ifdef MOIRA_CTA_TIMES
moira_status moira_set_cta_times(uint64_t *buf, int32_t max_launches)
{
    if (max_launches < 0 || (buf == nullptr && max_launches != 0)) return MOIRA_EINVAL;
    g_cta_times = reinterpret_cast<unsigned long long *>(buf);
    g_cta_launches = max_launches;
    return MOIRA_OK;
}
#endif

const char *moira_status_string(moira_status status)
{
    switch (status) {
    case MOIRA_OK: return "ok";
    case MOIRA_EINVAL: return "invalid argument";
    case MOIRA_EWORKSPACE: return "workspace missing, misaligned or too small";
    case MOIRA_ECUDA: return "CUDA runtime error";
    case MOIRA_EUNSUPPORTED: return "shape not supported by this library";
    }
    return "unknown status";
}

}  // extern "C"
