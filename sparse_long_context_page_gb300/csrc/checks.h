// Host-side argument checks shared by the C ABI's entry points (api.cu and
// noalloc.cu), so that every entry point rejects the same bad arguments the
// same way.
#pragma once

#include <stdint.h>

#include "../../include/moira.h"

namespace moira {

// Shape, batch and max_pages: MOIRA_EINVAL for nonsense, MOIRA_EUNSUPPORTED
// for sizes the kernels are not built for.
moira_status check_shape(const moira_shape *s);
moira_status check_batch(const moira_shape *s, int32_t batch, int32_t max_pages);

// Everything moira_select_ex checks except the workspace: the shape and
// batch as above, the summary format, the rule and its parameter, a finite
// positive sm_scale, non-null buffers, and q and the summaries on 16-byte
// boundaries.
moira_status check_select_args(const moira_shape *shape, int32_t fmt, const void *q, const void *summ,
                               const int32_t *page_table, const int32_t *seq_lens, int32_t batch,
                               int32_t max_pages, int32_t rule, float param, float sm_scale,
                               const int32_t *lists, const int32_t *lengths);

}  // namespace moira
