// prefill.cuh -- parameters of the causal partial-prefill kernel
// (prefill_umma.cu), shared with the host launcher (shkv_host.cu).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "shkv.h"

namespace shkv {

// Causal partial prefill of n_new appended tokens (prefill_umma.cu).
struct PrefillParams {
    const __nv_bfloat16 *q;      // [B, n_new, Hq, D]
    __nv_bfloat16 *out;          // [B, n_new, Hq, D]
    float *lse_out;              // [B, n_new, Hq] or null
    const int32_t *block_table;
    const int32_t *seq_lens;     // device copy (checked against lens)
    uint32_t *err;
    int32_t batch, n_new, hq, hkv, group, tpt, tiles;   // tiles per (request, head)
    int32_t page_size, max_pages, num_pages, stages;
    float scale_log2;
    int32_t lens[SHKV_MAX_BATCH];    // host copy of the lengths (with the new tokens)
    int32_t order[SHKV_MAX_BATCH];   // requests by length, longest first (CTA dispatch order)
};

}  // namespace shkv
