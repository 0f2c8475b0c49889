/*
 * moira_cta_times.h -- the load-balance build of the sparse-decode library
 * (libmoira_cta_times.so: the same sources compiled with MOIRA_CTA_TIMES).
 *
 * The self-planning attention gives every block of its fixed grid an equal
 * share of the kept pages ("MOIRA: Mass-Oriented Indexing with Ragged
 * Attention for Long-Context Decoding", abstract: the attention plans its
 * own work from the list lengths, so ragged batches stay balanced).  This
 * build records, per attention launch (k_attend or the single-launch
 * selection + attention), each block's start and end of its attention work
 * in %globaltimer nanoseconds, so the balance (max / mean block time) can be
 * measured.  libmoira.so has none of it.
 */
#ifndef MOIRA_CTA_TIMES_H
#define MOIRA_CTA_TIMES_H

#include "moira.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The next `max_launches` attention launches issued by this library write
 * (start, end) of every block of their grid (moira_attend_grid_blocks()
 * blocks) into consecutive slices of `buf`: launch i, block b at
 * buf[2 * (i * blocks + b)] and buf[2 * (i * blocks + b) + 1]; a block
 * without pages writes (0, 0).  buf is a DEVICE pointer of
 * 2 * blocks * max_launches uint64 words owned by the caller; the slices are
 * assigned when the launches are issued (so a captured graph keeps them).
 * NULL with 0 stops recording.  Host call; not thread-safe. */
MOIRA_API moira_status moira_set_cta_times(uint64_t *buf, int32_t max_launches);

#ifdef __cplusplus
}
#endif

#endif /* MOIRA_CTA_TIMES_H */
