// shard.cpp -- host-side division of a decode batch among replicas.
//
// PrefillShare (framework scope, Sec. 7): prefill and decode run in
// data-parallel pools of GPUs, each decode GPU serving its own requests over
// its own copy of the shared paged cache.  The decode step shards by request
// with no exchange step: every (request, KV head) unit is independent, so a
// replica needs only the pages of the requests it owns.  This file assigns
// requests to replicas so that each streams about the same number of unique
// KV bytes (the quantity that bounds the decode step), and is host code only
// (no CUDA).
#include <stdint.h>

#include <algorithm>
#include <numeric>
#include <vector>

#include "shkv.h"

extern "C" shkv_status shkv_partition_requests(int32_t batch, const int32_t *seq_lens, int32_t page_size,
                                               int32_t world_size, int32_t *owner, int64_t *rank_pages)
{
    if (batch < 0 || (batch > 0 && (!seq_lens || !owner)) || page_size < 1 || world_size < 1)
        return SHKV_ERR_INVALID_ARG;
    std::vector<int64_t> pages((size_t)batch);
    for (int32_t b = 0; b < batch; ++b) {
        if (seq_lens[b] < 0)
            return SHKV_ERR_INVALID_ARG;
        pages[(size_t)b] = ((int64_t)seq_lens[b] + page_size - 1) / page_size;
    }
    // Longest processing time first: requests by pages, descending (ties by
    // index), each to the replica holding the fewest pages so far (ties by
    // the lower rank).  Deterministic, so every rank computes the same
    // assignment from the same lengths without exchanging anything.
    std::vector<int32_t> order((size_t)batch);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t a, int32_t b) { return pages[(size_t)a] > pages[(size_t)b]; });
    std::vector<int64_t> load((size_t)world_size, 0);
    for (int32_t b : order) {
        int32_t best = 0;
        for (int32_t r = 1; r < world_size; ++r)
            if (load[(size_t)r] < load[(size_t)best])
                best = r;
        owner[b] = best;
        load[(size_t)best] += pages[(size_t)b];
    }
    if (rank_pages)
        for (int32_t r = 0; r < world_size; ++r)
            rank_pages[r] = load[(size_t)r];
    return SHKV_OK;
}
