// Local-window page recycling: the ring length a local buffer needs and the
// block-table rows that map a sequence's live pages into its ring.
//
// A local layer attends only the last `window` positions (hybrid attention with a
// 1024-token horizon, technique table of "Character.AI: inference optimization",
// section 03); everything older can be dropped.  Logical page k of a sequence is
// kept in ring slot k % ring.  A call touches, for the length hi after it,
//   decode:  [hi - window, hi)                          <= ceil((window - 1) / P) + 1 pages,
//   prefill: [max(0, hi - n + 1 - window), hi)          <= ceil((window + n - 1) / P) + 1 pages,
//   append:  [hi - n, hi)                               <= ceil((n - 1) / P) + 1 pages,
// all inside the last ceil((window + n - 1) / P) + 1 pages before ceil(hi / P), so a
// ring of that length never needs a slot that another live page occupies.
#include "cai.h"

extern "C" {

int32_t cai_ring_pages(int32_t window, int32_t page_size, int32_t max_new_tokens) {
  if (window < 1 || page_size < 1 || max_new_tokens < 1) return 0;
  const int64_t span = (int64_t)window + max_new_tokens - 1;
  const int64_t pages = (span + page_size - 1) / page_size + 1;
  return pages > 2147483647ll ? 0 : (int32_t)pages;
}

cai_status cai_ring_table_row(int32_t* row, int32_t max_pages_per_seq, const int32_t* ring_ids, int32_t ring,
                              int32_t hi, int32_t page_size) {
  if (!row || !ring_ids || ring < 1 || page_size < 1 || hi < 0 || max_pages_per_seq < 0) return CAI_ERR_INVALID_ARG;
  const int64_t top = ((int64_t)hi + page_size - 1) / page_size;  // pages holding [0, hi)
  if (top > max_pages_per_seq) return CAI_ERR_INVALID_ARG;
  const int64_t first = top > ring ? top - ring : 0;
  for (int64_t k = 0; k < max_pages_per_seq; ++k)
    row[k] = (k >= first && k < top) ? ring_ids[k % ring] : -1;
  return CAI_OK;
}

}  // extern "C"
