// tails.cuh -- the unit table of a decode with per-decoder tails in one pass
// (append_merge.cu builds it, shkv_host.cu launches it).
#pragma once

#include <stdint.h>

#include "shkv.h"

namespace shkv {

// Request b's unit: its S_b = ceil(L_b / P) shared pages, then for each
// decoder m its ceil(T_bm / P) tail pages.  unit_table[b * ustride + j] is
// the pool page of unit page j, unit_info the page's valid tokens (bits 0-7)
// and the decoder that attends it (bits 8-15; 0xff: all, a shared page).
struct TailsUnitParams {
    const int32_t *block_table;     // pool [max_batch, bt_stride]
    const int32_t *tail_table;      // tails [max_batch * n_models, tt_stride]
    int32_t *unit_table;            // [batch, ustride]
    uint32_t *unit_info;            // [batch, ustride]
    int32_t bt_stride, tt_stride, ustride, batch, n_models, page_size;
    int32_t wait_first;             // wait for the previous kernel before reading and writing
    int32_t shared_len[SHKV_MAX_BATCH];   // L_b
    int32_t tail_len[SHKV_MAX_BATCH];     // T_bm at b * n_models + m
};

}  // namespace shkv
