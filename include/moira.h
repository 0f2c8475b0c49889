/*
 * moira.h -- C ABI of the GB300 (sm_103a) sparse-decode library.
 *
 * The library implements the data-parallel hot path of MOIRA-style sparse
 * decoding described in "MOIRA: Mass-Oriented Indexing with Ragged Attention
 * for Long-Context Decoding" (arXiv 2610.04313), abstract:
 *   - per request, layer and KV head, at each decode step, a selection picks
 *     the fewest KV-cache pages whose estimated share of the attention adds
 *     up to at least gamma                              -> moira_select
 *   - an attention kernel then reads only the picked pages; each block works
 *     out on the device, from the list lengths alone, which pages it
 *     handles, so there is no host-side plan and a whole step can be
 *     captured as one CUDA graph                        -> moira_attend
 *   - the per-page estimate needs per-page metadata; following the
 *     mean-vector summaries named in "Faster Flash Decoding" (arXiv
 *     2609.00097), section 2, a page's summary is the bf16 mean of its keys
 *                                                       -> moira_update_summaries
 *
 * Estimator (the pages leave it open; this is the library's stated choice):
 *   kbar_p   = bf16 round-to-nearest-even of the mean of page p's keys
 *   s_{h,p}  = sm_scale * q_h . kbar_p            (query head h of the group)
 *   m_p      = (1/G) * sum_h softmax_p(s_{h,.})   (over the full pages)
 * Coverage: sort pages by (m_p descending, logical index ascending) and keep
 * the shortest prefix whose running sum is >= gamma; gamma >= 1 keeps every
 * page without estimating.  A partial last page (seq_len % page_size != 0)
 * has no summary yet; it is always kept and is the last list entry.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller allocates and owns every buffer.  The library never allocates,
 *     frees or synchronises inside moira_select / moira_attend /
 *     moira_decode_step and never reads device data back on the host there,
 *     so those calls can be captured in a CUDA graph (gamma and sm_scale are
 *     then fixed at capture time).
 *   - bf16 tensors are passed as raw pointers to IEEE bfloat16 values.
 *   - Layouts are dense, row-major, without padding.  Query head h reads KV
 *     head h / G with G = num_q_heads / num_kv_heads.
 *   - Host-side argument checks run first; on any error nothing is launched
 *     and a status other than MOIRA_OK is returned.
 *   - Problems only visible on the device (a physical page id outside the
 *     pool, a length out of range, a device wait that ran out) never trap:
 *     the kernel skips or clamps the offending item and ORs a MOIRA_DEV_*
 *     bit into the status word kept in the workspace; read it with
 *     moira_read_device_status().
 *   - Every device wait is bounded (2 s).  The first wait of a launch that
 *     runs out sets MOIRA_DEV_TIMEOUT, and from then on every wait of that
 *     launch, and of every later launch that starts while the bit is set,
 *     gives up at once, so a lost copy costs about one limit per step.  The
 *     results are then invalid: read and clear the status and call
 *     moira_workspace_init before the workspace is used again.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).
 */
#ifndef MOIRA_H
#define MOIRA_H

#include <stddef.h>
#include <stdint.h>

/* Only the functions declared here are exported from the library. */
#if defined(__GNUC__)
#define MOIRA_API __attribute__((visibility("default")))
#else
#define MOIRA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moira_stream_t;   /* identical to cudaStream_t */

typedef enum moira_status {
    MOIRA_OK = 0,
    MOIRA_EINVAL = 1,        /* an argument failed a host-side check; nothing launched */
    MOIRA_EWORKSPACE = 2,    /* workspace NULL, misaligned or smaller than required */
    MOIRA_ECUDA = 3,         /* a CUDA runtime call or a kernel launch failed */
    MOIRA_EUNSUPPORTED = 4   /* a shape this library does not implement (see moira_shape) */
} moira_status;

/* Bits of the device status word (sticky until cleared). */
#define MOIRA_DEV_BADPAGE 0x1u   /* a page id outside [0, num_phys_pages) was skipped */
#define MOIRA_DEV_BADLEN  0x2u   /* a seq_len or list length out of range was clamped */
#define MOIRA_DEV_TIMEOUT 0x4u   /* a bounded device wait ran out; results are invalid */

/* Limits of this library. */
#define MOIRA_HEAD_DIM 128               /* d */
#define MOIRA_PAGE_SIZE 16               /* S, tokens per page */
#define MOIRA_GROUP 4                    /* G = Hq / Hkv */
#define MOIRA_MAX_PAGES_PER_SEQ 16384    /* max_pages: 256k tokens per request */
#define MOIRA_MAX_UNITS 4096             /* batch * num_kv_heads */

/* Model / cache geometry.  This build requires head_dim == 128,
 * page_size == 16 and num_q_heads == 4 * num_kv_heads
 * (MOIRA_EUNSUPPORTED otherwise). */
typedef struct moira_shape {
    int32_t num_q_heads;      /* Hq */
    int32_t num_kv_heads;     /* Hkv */
    int32_t head_dim;         /* d */
    int32_t page_size;        /* S */
    int64_t num_phys_pages;   /* P: pages in ONE layer's pool */
} moira_shape;

/* Bytes of device workspace that moira_select / moira_attend /
 * moira_decode_step need for `batch` requests of at most `max_pages` pages,
 * on the CURRENT device (the attention grid is sized from its SM count).
 * Returns 0 if the arguments are invalid.  One workspace may serve every
 * layer of a step issued in order on one stream; concurrent calls need
 * separate workspaces. */
MOIRA_API size_t moira_workspace_bytes(const moira_shape *shape, int32_t batch, int32_t max_pages);

/* Zero the workspace (device status word and the self-resetting merge
 * counters must start at zero).  Call once after allocating it.  Enqueues a
 * memset on `stream`; returns MOIRA_ECUDA if that fails. */
MOIRA_API moira_status moira_workspace_init(void *workspace, size_t ws_bytes, moira_stream_t stream);

/* Page-summary formats.  The estimator reads one summary per (page, KV head).
 * MOIRA_SUMM_BF16 stores the mean key as bf16 [P][Hkv][d].  The low-bit
 * formats store the same mean key (taken in fp64, before any rounding) with
 * the symmetric mid-rise quantiser that "Faster Flash Decoding" (section
 * 3.1) uses for its low-bit key thumbnails, here with b = 8 or 2 bits:
 *   step   = max_i |mean_i| / (2^(b-1) - 1/2), rounded once to fp32
 *   code_i = floor(mean_i / step), clamped to [-2^(b-1), 2^(b-1) - 1]
 * and the summary stands for (code_i + 1/2) * step.  The quantiser has no
 * zero level, so every element keeps its sign.  A mean with a non-finite
 * element, an all-zero mean, or a step that rounds to 0 gets step 0 and
 * codes 0.
 * Low-bit layout: one record of moira_summary_page_bytes() bytes per
 * physical page.  The record holds the KV heads in groups of gh = min(Hkv, 4)
 * consecutive heads, group after group, and each group is
 *   bytes [0, gh*cb)            codes, head jj of the group at [jj*cb, (jj+1)*cb),
 *                               cb = d*b/8
 *                               Q8: byte i = code of element i (int8)
 *                               Q2: element i in bits 2*(i%4)+1 .. 2*(i%4) of
 *                                   byte i/4, stored as code + 2 (0..3)
 *   bytes [gh*cb, gh*cb + 4*gh) fp32 step of each head of the group
 *   then zero bytes up to gh*cb + 16
 * so the summaries of one group of heads are one contiguous, 16-byte aligned
 * run.  At Hkv = 8 a page's summaries take 2048 (BF16), 1056 (Q8) or 288 (Q2)
 * bytes. */
typedef enum {
    MOIRA_SUMM_BF16 = 0,
    MOIRA_SUMM_Q8 = 1,
    MOIRA_SUMM_Q2 = 2
} moira_summ_format;

/* Bytes of one physical page's summaries (all KV heads) in `format`, i.e.
 * one layer's summary buffer holds num_phys_pages times this.  0 if the shape
 * or the format is invalid. */
MOIRA_API size_t moira_summary_page_bytes(const moira_shape *shape, int32_t format);

/* Page summaries, made when a page fills (the per-page metadata the "MOIRA"
 * abstract's estimate needs; estimator form: mean vectors, "Faster Flash
 * Decoding" section 2).
 * For each listed physical page p and KV head j:
 *   summ[p][j][:] = bf16_rne( mean over the S tokens of k_pool[p][j][:][:] ),
 * accumulated in fp64 so that the mean is rounded once.
 *   k_pool     : bf16 [P][Hkv][S][d]   one layer's key pool (read)
 *   summ       : bf16 [P][Hkv][d]      that layer's summaries (written for
 *                                      the listed pages only)
 *   phys_pages : int32 [n]             physical page ids; ids outside [0, P)
 *                                      are skipped (MOIRA_DEV_BADPAGE)
 * Not part of the decode step: call it when pages fill or after prefill. */
MOIRA_API moira_status moira_update_summaries(const moira_shape *shape, const void *k_pool, void *summ,
                                    const int32_t *phys_pages, int32_t n, moira_stream_t stream);

/* moira_update_summaries in any summary format (moira_summ_format): `summ`
 * is that layer's summary buffer, num_phys_pages * moira_summary_page_bytes()
 * bytes, 16-byte aligned.  MOIRA_SUMM_BF16 is exactly moira_update_summaries.
 * An unknown format returns MOIRA_EINVAL. */
MOIRA_API moira_status moira_update_summaries_ex(const moira_shape *shape, int32_t format, const void *k_pool,
                                       void *summ, const int32_t *phys_pages, int32_t n,
                                       moira_stream_t stream);

/* Append one token per request to one layer's paged KV cache and keep the
 * page summaries current: moira_update_summaries for every page the append
 * fills, fused with the append a serving loop does every step (the pages
 * leave the append itself to the serving system).  Request r's new token is
 * token seq_lens[r] - 1, i.e. seq_lens counts it, as moira_select and
 * moira_attend expect afterwards.  Its key and value go to slot
 * (seq_lens[r]-1) % S of logical page (seq_lens[r]-1) / S; when that is the
 * page's last slot, summ[page][j] is recomputed exactly as
 * moira_update_summaries would.
 *   k_new, v_new : bf16 [batch][Hkv][d]        the new token's keys / values
 *   k_pool, v_pool : bf16 [P][Hkv][S][d]       one layer's pools (written)
 *   summ       : bf16 [P][Hkv][d]              that layer's summaries (written
 *                                              for pages that fill)
 *   page_table : int32 [batch][max_pages]      logical -> physical page
 *   seq_lens   : int32 [batch]                 tokens after the append; 0
 *                                              appends nothing for that request
 * A length beyond max_pages * S or a page id outside [0, P) skips that
 * request (no workspace, so nothing is recorded).  All buffers device,
 * 16-byte aligned. */
MOIRA_API moira_status moira_append_kv(const moira_shape *shape, const void *k_new, const void *v_new,
                             void *k_pool, void *v_pool, void *summ, const int32_t *page_table,
                             const int32_t *seq_lens, int32_t batch, int32_t max_pages,
                             moira_stream_t stream);

/* moira_append_kv with the summaries of filled pages written in `format`
 * (as moira_update_summaries_ex would write them). */
MOIRA_API moira_status moira_append_kv_ex(const moira_shape *shape, int32_t format, const void *k_new,
                                const void *v_new, void *k_pool, void *v_pool, void *summ,
                                const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                                int32_t max_pages, moira_stream_t stream);

/* The coverage rule of the "MOIRA" abstract (the fewest pages whose estimated
 * attention share reaches gamma), for every (request, KV head) of one layer.
 *   q          : bf16 [batch][Hq][d]          this layer's queries
 *   summ       : bf16 [P][Hkv][d]             this layer's page summaries
 *   page_table : int32 [batch][max_pages]     logical -> physical page
 *   seq_lens   : int32 [batch]                tokens per request, including
 *                                             the current one (0 allowed)
 *   gamma      : (0, 1]; 1 keeps every page (dense) without estimating
 *   sm_scale   : score scale, normally 1/sqrt(d)
 *   lists      : int32 [batch][Hkv][max_pages] out: physical ids of the kept
 *                pages in ascending logical order, the partial tail page (if
 *                any) last; entries past `lengths` are left untouched
 *   lengths    : int32 [batch][Hkv] out
 * Equal masses are taken lower logical index first.  If rounding keeps the
 * total estimated mass below gamma, every page is kept. */
MOIRA_API moira_status moira_select(const moira_shape *shape, const void *q, const void *summ,
                          const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                          int32_t max_pages, float gamma, float sm_scale, int32_t *lists,
                          int32_t *lengths, void *workspace, size_t ws_bytes,
                          moira_stream_t stream);

/* Page rules for moira_select_rule. */
typedef enum {
    MOIRA_RULE_COVERAGE = 0,  /* smallest set reaching mass gamma ("MOIRA" abstract); param = gamma */
    MOIRA_RULE_TOPK = 1,      /* fixed budget ("Faster Flash Decoding" section 1, figure 1 (a)):
                                 the k heaviest full pages, equal masses lower index first;
                                 param = k, a whole number in [0, 2^24] */
    MOIRA_RULE_TOPDELTA = 2   /* relative threshold to the maximum ("Faster Flash Decoding"
                                 section 1, figure 1 (c); its formula is cut from the page, read
                                 as): every full page with mass >= delta * the unit's largest
                                 mass; param = delta in (0, 1] */
} moira_rule;

/* moira_select with the page rule chosen by `rule` (see moira_rule).  The
 * estimator, the partial tail page (always kept, last), the list order, the
 * buffers, the workspace and the errors are those of moira_select;
 * MOIRA_RULE_COVERAGE with param = gamma is exactly moira_select.  A `param`
 * outside the rule's range returns MOIRA_EINVAL and launches nothing.  The
 * rules let a caller compare selections that read the same number of bytes. */
MOIRA_API moira_status moira_select_rule(const moira_shape *shape, const void *q, const void *summ,
                               const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                               int32_t max_pages, int32_t rule, float param, float sm_scale,
                               int32_t *lists, int32_t *lengths, void *workspace, size_t ws_bytes,
                               moira_stream_t stream);

/* moira_select_rule reading summaries in `format` (moira_summ_format): the
 * estimator takes the summary's value, (code + 1/2) * step for the low-bit
 * formats, in place of the bf16 mean key; everything else is unchanged.
 * MOIRA_SUMM_BF16 is exactly moira_select_rule. */
MOIRA_API moira_status moira_select_ex(const moira_shape *shape, int32_t format, const void *q,
                             const void *summ, const int32_t *page_table, const int32_t *seq_lens,
                             int32_t batch, int32_t max_pages, int32_t rule, float param,
                             float sm_scale, int32_t *lists, int32_t *lengths, void *workspace,
                             size_t ws_bytes, moira_stream_t stream);

/* Self-planning ragged attention (the "MOIRA" abstract: blocks plan their own
 * work from the list lengths on the device, which keeps the step graph-
 * capturable).  A fixed grid (a multiple of
 * the SM count) splits the concatenated lists into equal page ranges; each
 * block finds its range from a device-side scan of `lengths`, computes
 * online-softmax partials per list segment, and the last block to finish a
 * list merges its partials by log-sum-exp (sequence-split decoding,
 * "Faster Flash Decoding" section 2).
 *   q          : bf16 [batch][Hq][d]
 *   k_pool     : bf16 [P][Hkv][S][d]   this layer's keys   (16-byte aligned)
 *   v_pool     : bf16 [P][Hkv][S][d]   this layer's values (16-byte aligned)
 *   lists, lengths : as produced by moira_select (any lists that follow the
 *                same contract are accepted: the last entry of a list holds
 *                seq_len % S valid tokens when that is non-zero)
 *   seq_lens   : int32 [batch]
 *   out        : fp32 [batch][Hq][d] out: softmax(sm_scale q K^T) V over the
 *                listed tokens; zero for an empty list
 * Computes in bf16 x bf16 -> fp32 on the tensor cores with fp32 softmax. */
MOIRA_API moira_status moira_attend(const moira_shape *shape, const void *q, const void *k_pool,
                          const void *v_pool, const int32_t *lists, const int32_t *lengths,
                          const int32_t *seq_lens, int32_t batch, int32_t max_pages,
                          float sm_scale, float *out, void *workspace, size_t ws_bytes,
                          moira_stream_t stream);

/* One layer's selection and attention: exactly the lists and lengths of
 * moira_select, and the output of moira_attend over them (within the
 * attention tolerance: the fp32 summation order may differ).  Arguments as
 * in those two calls; out: fp32 [batch][Hq][d].
 * For small batches (fewer than 64 (request, KV head) lists, and at most
 * 512 pages per block when each list's pages are split over
 * grid / lists blocks of the attention grid: about 19k pages per request at
 * 8 lists on 152 SMs) the selection is spread over the whole attention grid
 * and runs in the same launch as the attention (the "MOIRA" abstract's
 * self-planning attention with its selection cost taken off the critical
 * path): after the score kernel, one launch whose blocks meet at barriers
 * inside it, so every block of the grid must be resident at once (checked
 * once per device; another kernel that holds SMs for longer than the device
 * wait limit makes the launch report MOIRA_DEV_TIMEOUT).  Larger batches run
 * moira_select then moira_attend. */
MOIRA_API moira_status moira_select_attend(const moira_shape *shape, const void *q, const void *summ,
                                 const void *k_pool, const void *v_pool, const int32_t *page_table,
                                 const int32_t *seq_lens, int32_t batch, int32_t max_pages, float gamma,
                                 float sm_scale, int32_t *lists, int32_t *lengths, float *out,
                                 void *workspace, size_t ws_bytes, moira_stream_t stream);

/* moira_select_attend reading summaries in `format` (moira_summ_format), as
 * moira_select_ex does with the coverage rule.  MOIRA_SUMM_BF16 is exactly
 * moira_select_attend. */
MOIRA_API moira_status moira_select_attend_ex(const moira_shape *shape, int32_t format, const void *q,
                                    const void *summ, const void *k_pool, const void *v_pool,
                                    const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                                    int32_t max_pages, float gamma, float sm_scale, int32_t *lists,
                                    int32_t *lengths, float *out, void *workspace, size_t ws_bytes,
                                    moira_stream_t stream);

/* The page-scoring kernel of moira_select_ex alone: the logits of every
 * (request, KV head, full page) against the summaries, reduced to per-chunk
 * softmax statistics in the workspace (the estimator's first half; the
 * "MOIRA" abstract's estimated mass needs them).  Its results are internal
 * to the workspace; the call exists to time how a layer's work splits
 * between scoring and the rest.  Arguments and errors as moira_select_ex. */
MOIRA_API moira_status moira_score_ex(const moira_shape *shape, int32_t format, const void *q, const void *summ,
                            const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                            int32_t max_pages, float sm_scale, void *workspace, size_t ws_bytes,
                            moira_stream_t stream);

/* The coverage selection of moira_select in one launch, one thread-block
 * cluster of 16 or 8 blocks per list, the blocks exchanging the chunk
 * statistics, histogram slices, candidates and kept counts through
 * distributed shared memory (NEXT-1's score + select fusion).  Same
 * arguments, results and errors as moira_select, whose lists and lengths it
 * gives bit for bit; it is slower on GB300 at batch 1 (21 against 15 us per
 * 128k layer), so neither moira_select nor the decode step uses it.  Returns
 * MOIRA_EUNSUPPORTED, launching nothing, when the device cannot hold every
 * list's cluster at once or max_pages needs more than two rounds of chunks
 * per block (moira_select_cluster_size).  gamma >= 1 runs moira_select's
 * dense path. */
MOIRA_API moira_status moira_select_clustered(const moira_shape *shape, const void *q, const void *summ,
                                    const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                                    int32_t max_pages, float gamma, float sm_scale, int32_t *lists,
                                    int32_t *lengths, void *workspace, size_t ws_bytes, moira_stream_t stream);

/* The cluster size (16 or 8) moira_select_clustered takes for these sizes on
 * the current device, or 0 when it returns MOIRA_EUNSUPPORTED (or the
 * arguments are invalid). */
MOIRA_API int32_t moira_select_cluster_size(const moira_shape *shape, int32_t batch, int32_t max_pages);

/* 1 if moira_select_attend takes the single-launch form for these sizes on
 * the current device, 0 if it runs moira_select then moira_attend (or the
 * arguments are invalid).  The decode step always runs moira_select then
 * moira_attend per layer. */
MOIRA_API int32_t moira_select_attend_is_fused(const moira_shape *shape, int32_t batch, int32_t max_pages);

/* One whole decode-attention step: for layer l = 0 .. num_layers-1,
 * moira_select then moira_attend on that layer's slices, in order on one
 * stream (the per-layer calls above, looped on the host).  The output
 * equals moira_select_attend's per layer bit for bit (same lists, same
 * attention plan and data path).
 *   q_all      : bf16 [L][batch][Hq][d]
 *   k_pool_all, v_pool_all : bf16 [L][P][Hkv][S][d]
 *   summ_all   : bf16 [L][P][Hkv][d]
 *   lists      : int32 [batch][Hkv][max_pages]  scratch, reused per layer
 *   lengths_all: int32 [L][batch][Hkv] out (every layer's list lengths)
 *   out_all    : fp32 [L][batch][Hq][d] out
 * page_table and seq_lens must not change until the step's work is done:
 * from layer 1 on, the score kernel reads them while the previous layer's
 * attention is still finishing. */
MOIRA_API moira_status moira_decode_step(const moira_shape *shape, int32_t num_layers, const void *q_all,
                               const void *k_pool_all, const void *v_pool_all,
                               const void *summ_all, const int32_t *page_table,
                               const int32_t *seq_lens, int32_t batch, int32_t max_pages,
                               float gamma, float sm_scale, int32_t *lists, int32_t *lengths_all,
                               float *out_all, void *workspace, size_t ws_bytes,
                               moira_stream_t stream);

/* moira_decode_step with any summary format and page rule: per layer
 * moira_select_ex(format, rule, param) then moira_attend.  summ_all holds
 * the layers' summary buffers back to back, num_phys_pages *
 * moira_summary_page_bytes() bytes each. */
MOIRA_API moira_status moira_decode_step_ex(const moira_shape *shape, int32_t format, int32_t num_layers,
                                  const void *q_all, const void *k_pool_all,
                                  const void *v_pool_all, const void *summ_all,
                                  const int32_t *page_table, const int32_t *seq_lens,
                                  int32_t batch, int32_t max_pages, int32_t rule, float param,
                                  float sm_scale, int32_t *lists, int32_t *lengths_all,
                                  float *out_all, void *workspace, size_t ws_bytes,
                                  moira_stream_t stream);

/* The same step with the per-step inputs and outputs in HOST memory:
 * q_host (bf16 [L][batch][Hq][d]) is copied to the device staging buffer
 * q_dev, the step runs, and out_dev is copied back to out_host (fp32
 * [L][batch][Hq][d]).  Copies are cudaMemcpyAsync on `stream` (pinned host
 * memory makes them asynchronous); the call does not synchronise. */
MOIRA_API moira_status moira_decode_step_host(const moira_shape *shape, int32_t num_layers,
                                    const void *q_host, void *q_dev, const void *k_pool_all,
                                    const void *v_pool_all, const void *summ_all,
                                    const int32_t *page_table, const int32_t *seq_lens,
                                    int32_t batch, int32_t max_pages, float gamma, float sm_scale,
                                    int32_t *lists, int32_t *lengths_all, float *out_dev,
                                    float *out_host, void *workspace, size_t ws_bytes,
                                    moira_stream_t stream);

/* The coverage selection of moira_select for callers that cannot allocate
 * device memory (a plug-in handed only its input and output buffers, a host
 * runtime whose device memory belongs to another allocator, or a decode loop
 * that must never call cudaMalloc).  The paper has no counterpart: it is a
 * deployment variant of moira_select.  Arguments and results are those of
 * moira_select without the workspace.  Its scratch (page weights and
 * per-chunk softmax normalisers, about 4*batch*Hq*max_pages bytes) lives in
 * a 4 MiB array compiled into the library, which every GPU that loads the
 * library holds until the process exits; sizes that need more return
 * MOIRA_EUNSUPPORTED and launch nothing.  Arguments are checked as
 * moira_select checks them (same codes).  The call runs on the current
 * device: `stream` must belong to it (else MOIRA_EINVAL, nothing launched).
 * The first call on a device looks up the array's device address with that
 * device current, so make it before any stream capture.  All calls share the array: calls that overlap on the
 * GPU (different streams, or a call still running when the next starts on
 * another stream) race; calls in order on one stream do not.  Device-side
 * range problems are skipped or clamped as in moira_select, but the status
 * word is internal and not reported.  Never calls cudaMalloc or cudaFree. */
MOIRA_API moira_status moira_select_noalloc(const moira_shape *shape, const void *q, const void *summ,
                                  const int32_t *page_table, const int32_t *seq_lens,
                                  int32_t batch, int32_t max_pages, float gamma, float sm_scale,
                                  int32_t *lists, int32_t *lengths, moira_stream_t stream);

/* Diagnostic of the device-side failure path: launches one block that waits,
 * exactly as the kernels' mbarrier waits do, on a barrier nothing will ever
 * complete, gives up after `limit_ns` nanoseconds (1 .. 10^10) and ORs
 * MOIRA_DEV_TIMEOUT into the workspace status word.  Lets a caller check that
 * a wait that runs out is reported through moira_read_device_status and
 * leaves the context usable.  No paper counterpart. */
MOIRA_API moira_status moira_diag_wait_timeout(void *workspace, size_t ws_bytes, uint64_t limit_ns,
                                     moira_stream_t stream);

/* Diagnostic of the give-up rule of the device waits: one block waits on
 * `n_waits` (1 .. 4096) barriers that nothing completes, one after the
 * other, the way the kernels wait: the first wait runs out after `limit_ns`
 * (1 .. 10^10) and sets MOIRA_DEV_TIMEOUT, and every later wait of the block
 * gives up at once, so the launch takes about one limit, not n_waits.  No
 * paper counterpart. */
MOIRA_API moira_status moira_diag_wait_chain(void *workspace, size_t ws_bytes, uint64_t limit_ns, int32_t n_waits,
                                   moira_stream_t stream);

/* Diagnostic of the inter-block barrier of moira_select_attend: `blocks`
 * (1 .. SM count) blocks meet at a barrier sized for one block more, so it
 * never completes; each block gives up after `limit_ns` and sets
 * MOIRA_DEV_TIMEOUT.  Uses (and clears) bytes 128..255 of the workspace.
 * No paper counterpart. */
MOIRA_API moira_status moira_diag_barrier_timeout(void *workspace, size_t ws_bytes, uint64_t limit_ns, int32_t blocks,
                                        moira_stream_t stream);

/* Synchronise `stream`, copy the device status word (MOIRA_DEV_* bits) to
 * *status_out (HOST pointer) and clear it when `clear` is non-zero.  A host
 * call: never issue it while `stream` is being captured. */
MOIRA_API moira_status moira_read_device_status(void *workspace, size_t ws_bytes, uint32_t *status_out,
                                      int32_t clear, moira_stream_t stream);

/* Thread blocks of the attention grid on the current device (a multiple of
 * its SM count); a property used by tests and benchmarks. */
MOIRA_API int32_t moira_attend_grid_blocks(void);

/* Static description of a status code. */
MOIRA_API const char *moira_status_string(moira_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOIRA_H */
