// decode_common.cuh -- pieces shared by the decode kernels: the split plan
// walk (segments of (request, KV head) units inside a CTA's chunk range),
// the shared-memory context and barrier addresses, and the TMA producer warp
// that streams a CTA's K/V pages and query rows into the mbarrier ring.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "shkv_device.cuh"

namespace shkv {
namespace detail {

constexpr float kLn2 = 0.6931471805599453f;

struct Segment {
    int b, g, pages_b, p0, p1;
    int64_t unit_begin, unit_end, seg_begin, seg_end;
};

// Chunk index -> (request, head, page) and the segment it starts, clipped to
// the CTA's range end.
__device__ __forceinline__ Segment locate(const DecodeParams &p, int64_t idx, int64_t cta_end)
{
    int lo = 0, hi = p.batch;
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if ((int64_t)p.hkv * p.page_prefix[mid] <= idx)
            lo = mid;
        else
            hi = mid;
    }
    Segment s;
    s.b = lo;
    s.pages_b = p.page_prefix[lo + 1] - p.page_prefix[lo];
    const int64_t base = (int64_t)p.hkv * p.page_prefix[lo];
    const int64_t rem = idx - base;
    s.g = (int)(rem / s.pages_b);
    s.p0 = (int)(rem - (int64_t)s.g * s.pages_b);
    s.unit_begin = base + (int64_t)s.g * s.pages_b;
    s.unit_end = s.unit_begin + s.pages_b;
    s.seg_begin = idx;
    s.seg_end = s.unit_end < cta_end ? s.unit_end : cta_end;
    s.p1 = s.p0 + (int)(s.seg_end - idx);
    return s;
}

// Successor of a segment that ended at its unit's end: the next (request,
// head) unit, from its first page, clipped to the CTA's range end.  Requests
// without pages (empty per-decoder tails) own no chunks and are stepped over;
// the caller only asks while chunks remain in its range, so one exists.
__device__ __forceinline__ Segment next_segment(const DecodeParams &p, const Segment &prev, int64_t cta_end)
{
    Segment s;
    s.g = prev.g + 1;
    s.b = prev.b;
    if (s.g == p.hkv) {
        s.g = 0;
        s.b = prev.b + 1;
        while (s.b + 1 < p.batch && p.page_prefix[s.b + 1] == p.page_prefix[s.b])
            ++s.b;
    }
    s.pages_b = p.page_prefix[s.b + 1] - p.page_prefix[s.b];
    s.unit_begin = prev.unit_end;
    s.unit_end = s.unit_begin + s.pages_b;
    s.seg_begin = s.unit_begin;
    s.seg_end = s.unit_end < cta_end ? s.unit_end : cta_end;
    s.p0 = 0;
    s.p1 = (int)(s.seg_end - s.seg_begin);
    return s;
}

__device__ __forceinline__ int64_t cta_start(const DecodeParams &p, int c) { return p.cta_cut[c]; }

// CTA whose range [cta_cut[c], cta_cut[c+1]) holds chunk idx.
__device__ __forceinline__ int cta_of(const DecodeParams &p, int64_t idx)
{
    int lo = 0, hi = p.num_ctas;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (p.cta_cut[mid] <= idx)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Window load of the unit table (page ids) or of page_info: entry j of
// request b's row, -1 past the segment.
__device__ __forceinline__ int unit_entry(const int32_t *table, const DecodeParams &p, int b, int j, int jend)
{
    return j < jend ? __ldg(table + (int64_t)b * p.max_pages + j) : -1;
}

// Cached length of request b, from the split plan (the host's copy).
__device__ __forceinline__ int plan_len(const DecodeParams &p, const Segment &s)
{
    return (s.pages_b - 1) * p.page_size + (int)p.last_fill[s.b];
}

// Partial slot written by CTA c for its piece of the unit starting at
// unit_begin: slot 0 if the piece opens the CTA's range, else slot 1.
__device__ __forceinline__ int piece_slot(const DecodeParams &p, int c, int64_t unit_begin)
{
    const int64_t st = cta_start(p, c);
    return 2 * c + (unit_begin <= st ? 0 : 1);
}

__device__ __forceinline__ int q_row(const DecodeParams &p, int g, int r)
{
    const int m = r / p.group, j = r - (r / p.group) * p.group;
    return m * p.hq + g * p.group + j;
}

struct Ctx {
    uint8_t *smem;
    DecodeSmem lay;
    uint32_t base;          // shared-space address of smem
    volatile uint32_t *abort_flag;
    uint32_t *bcast;
    int64_t cta_begin, cta_end;
};

__device__ __forceinline__ uint32_t full_bar(const Ctx &c, int s) { return c.base + c.lay.bars + 8u * s; }
__device__ __forceinline__ uint32_t empty_bar(const Ctx &c, int s, int stages)
{
    return c.base + c.lay.bars + 8u * (stages + s);
}
__device__ __forceinline__ uint32_t qfull_bar(const Ctx &c, int i, int stages)
{
    return c.base + c.lay.bars + 8u * (2 * stages + i);
}
__device__ __forceinline__ uint32_t qempty_bar(const Ctx &c, int i, int stages)
{
    return c.base + c.lay.bars + 8u * (2 * stages + 2 + i);
}

// ---------------------------------------------------------------------------
// producer warp
// ---------------------------------------------------------------------------
// Stage j of a segment holds the kStageTokens logical tokens starting at
// p0*P + j*kStageTokens, as one or two row-blocks of BR = min(P, kStageTokens)
// rows, each row-block inside one page.
// Run by the producer warp before it waits for the previous grid: prefetch
// into L2 the K/V row-blocks of this CTA's first ring-full of stages (up to
// 32 pages of its first segment), so that its first copies after the wait
// hit L2 instead of waiting on DRAM.  The block-table entries are read
// through L2 only and may be stale (a preceding kernel may still be writing
// them): they are used for nothing but these prefetches, and an id outside
// the pool is skipped.
template <int D>
__device__ void warm_l2(const CUtensorMap *tmK, const CUtensorMap *tmV, const DecodeParams &p, const Ctx &c)
{
    const int lane = threadIdx.x & 31;
    const Segment s = locate(p, c.cta_begin, c.cta_end);
    const int P = p.page_size;
    const int ring_pages = p.stages * kStageTokens / P;
    const int pages = s.p1 - s.p0 < ring_pages ? s.p1 - s.p0 : ring_pages;
    if (lane < pages) {
        const int id = __ldcg(p.block_table + (int64_t)s.b * p.max_pages + s.p0 + lane);
        if (id >= 0 && id < p.num_pages)
            for (int rb = 0; rb < P; rb += p.box_rows) {
                const int y = (id * p.hkv + s.g) * P + rb;
                tma_prefetch_3d_row(tmK, y);
                tma_prefetch_3d_row(tmV, y);
            }
    }
}

// FUSED: the units are fused per-decoder tails (DecodeParams::page_info).
template <int D, bool FUSED>
__device__ void producer(const CUtensorMap *tmK, const CUtensorMap *tmV, const DecodeParams &p,
                         const Ctx &c)
{
    constexpr int TT = kStageTokens;
    const int lane = threadIdx.x & 31;
    const int stages = p.stages;
    const int P = p.page_size;
    const int BR = p.box_rows;
    const int RB = TT / BR;                        // row-blocks per stage (1 or 2)
    const int log2P = 31 - __clz(P);
    const uint32_t rb_bytes_kv = 2u * (uint32_t)BR * D * 2u;
    const uint64_t pol = l2_evict_first_policy();
    if (lane == 0) {
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
    }

    bool alive = true;
    int kbase = 0, seg = 0;
    int last_issued_stage = -1;     // highest stage index with copies issued
    int q_issued[2] = {-1, -1};     // segment whose Q was last issued per buffer
    Segment s = locate(p, c.cta_begin, c.cta_end);
    // first block-table window of the current segment, prefetched one
    // segment ahead
    const int32_t *info_tab = reinterpret_cast<const int32_t *>(p.page_info);
    constexpr bool fused = FUSED;
    int pre = unit_entry(p.block_table, p, s.b, s.p0 + lane, s.p1);
    int pre_i = fused ? unit_entry(info_tab, p, s.b, s.p0 + lane, s.p1) : -1;
    for (;;) {
        const bool has_next = s.seg_end < c.cta_end;
        Segment sn;
        int pre_next = -1, pre_next_i = -1;
        if (has_next) {
            sn = next_segment(p, s, c.cta_end);
            pre_next = unit_entry(p.block_table, p, sn.b, lane, sn.p1);
            if (fused)
                pre_next_i = unit_entry(info_tab, p, sn.b, lane, sn.p1);
        }
        // device copy of the length, checked at the end of the segment
        // (a unit of fused tails is not one sequence: nothing to check)
        const int dev_len = (lane == 0 && !fused) ? __ldg(p.seq_lens + s.b) : 0;
        // --- query rows of this (b, g): N bulk copies of G contiguous rows
        const int qb = seg & 1;
        if (alive) {
            bool ok = mbar_wait_bounded(qempty_bar(c, qb, stages), ((seg >> 1) & 1) ^ 1, c.abort_flag, p.err);
            alive = __all_sync(0xffffffffu, ok);
        }
        if (alive && lane == 0) {
            const uint32_t rows_bytes = (uint32_t)p.group * D * 2u;
            mbar_arrive_expect_tx(qfull_bar(c, qb, stages), rows_bytes * p.n_models);
            const __nv_bfloat16 *qsrc = p.q + ((int64_t)s.b * p.n_models * p.hq + (int64_t)s.g * p.group) * D;
            const uint32_t qdst = c.base + c.lay.qbuf + qb * c.lay.qbuf_bytes;
            for (int m = 0; m < p.n_models; ++m)
                bulk_load(qdst + m * rows_bytes, qsrc + (int64_t)m * p.hq * D, rows_bytes,
                          qfull_bar(c, qb, stages));
            q_issued[qb] = seg;
        }
        // --- K/V row-blocks of the segment
        const int tok_end = s.p1 * P;
        const int nst = (tok_end - s.p0 * P + TT - 1) / TT;
        const int32_t *btrow = p.block_table + (int64_t)s.b * p.max_pages;
        int w0 = s.p0;                                   // block-table window [w0, w0+32)
        int cur = pre, cur_i = pre_i;
        int nxt = (w0 + 32 + lane < s.p1) ? __ldg(btrow + w0 + 32 + lane) : -1;
        int nxt_i = fused ? unit_entry(info_tab, p, s.b, w0 + 32 + lane, s.p1) : -1;
        // Lane 4*sub + 2*rb + kv copies row-block rb of K (kv = 0) or V
        // (kv = 1) for stage j + sub of this iteration.
        const int sub = lane >> 2;
        const int my_rb = (lane >> 1) & 1;
        const int my_kv = lane & 1;
        for (int j = 0; j < nst; j += kStagesPerIssue) {
            const int jj = j + sub;
            const bool in_iter = sub < kStagesPerIssue && jj < nst;
            const int k = kbase + jj;
            const int slot = k % stages;
            const int tok0 = s.p0 * P + jj * TT;
            // window of block-table entries for the first page of this iteration
            const int pg_first = (s.p0 * P + j * TT) >> log2P;
            if (pg_first >= w0 + 32) {
                w0 += 32;
                cur = nxt;
                nxt = (w0 + 32 + lane < s.p1) ? __ldg(btrow + w0 + 32 + lane) : -1;
                if (fused) {
                    cur_i = nxt_i;
                    nxt_i = unit_entry(info_tab, p, s.b, w0 + 32 + lane, s.p1);
                }
            }
            const int my_tok = tok0 + my_rb * BR;
            const int my_pg = my_tok >> log2P;
            const int my_id = __shfl_sync(0xffffffffu, cur, (my_pg - w0) & 31);
            int my_info = 0, rb1_info = 0;
            if (fused) {
                my_info = __shfl_sync(0xffffffffu, cur_i, (my_pg - w0) & 31);
                rb1_info = __shfl_sync(0xffffffffu, my_info, (lane + 2) & 31);   // row-block 1, seen by lane 4*sub
            }
            bool ok = true;
            if (alive && in_iter)           // the 4 lanes of each stage poll its slot together
                ok = mbar_wait_bounded(empty_bar(c, slot, stages), ((k / stages) & 1) ^ 1, c.abort_flag, p.err);
            alive = alive && __all_sync(0xffffffffu, ok);
            const bool my_valid = in_iter && my_rb < RB && my_tok < tok_end && my_id >= 0 && my_id < p.num_pages;
            const uint32_t vmask = __ballot_sync(0xffffffffu, my_valid && my_kv == 0);
            if (alive && in_iter && (lane & 3) == 0) {
                const uint32_t bits = vmask >> lane;     // bit 0: rb 0, bit 2: rb 1
                uint32_t mask = 0;
                for (int rb = 0; rb < RB; ++rb) {
                    if ((bits >> (2 * rb)) & 1u)
                        mask |= 1u << rb;
                    else if (tok0 + rb * BR < tok_end)
                        atomicOr(p.err, SHKV_ERRF_PAGE_OOB);
                }
                volatile uint32_t *meta = reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.meta) + slot * kMetaWords;
                if (fused) {
                    meta[1] = (uint32_t)my_info;
                    meta[2] = (uint32_t)rb1_info;
                }
                meta[0] = mask | ((uint32_t)k << 8);   // valid row-blocks + stage tag
                mbar_arrive_expect_tx(full_bar(c, slot), (uint32_t)__popc(mask) * rb_bytes_kv);
            }
            __syncwarp();
            if (alive && my_valid) {
                const uint32_t dst = c.base + c.lay.ring + (uint32_t)slot * c.lay.stage_bytes +
                                     (uint32_t)my_kv * (TT * D * 2) + (uint32_t)my_rb * (BR * D * 2);
                const int y = (my_id * p.hkv + s.g) * P + (my_tok & (P - 1));
                tma_load_3d_row(dst, my_kv ? tmV : tmK, y, full_bar(c, slot), pol);
            }
            if (alive) {
                const int last = kbase + (j + kStagesPerIssue < nst ? j + kStagesPerIssue : nst) - 1;
                last_issued_stage = last;
            }
            __syncwarp();
        }
        if (lane == 0 && !fused && dev_len != plan_len(p, s))
            atomicOr(p.err, SHKV_ERRF_SEQ_LEN);
        kbase += nst;
        ++seg;
        if (!has_next)
            break;
        s = sn;
        pre = pre_next;
        pre_i = pre_next_i;
    }
    // After an abort, wait (bounded) for every copy this CTA still has in
    // flight so no TMA write lands after the CTA exits.
    if (!alive && lane == 0) {
        for (int k = last_issued_stage - stages + 1; k <= last_issued_stage; ++k)
            if (k >= 0)
                mbar_drain_bounded(full_bar(c, k % stages), (uint32_t)((k / stages) & 1));
        for (int i = 0; i < 2; ++i)
            if (q_issued[i] >= 0)
                mbar_drain_bounded(qfull_bar(c, i, stages), (uint32_t)((q_issued[i] >> 1) & 1));
    }
}

}  // namespace detail
}  // namespace shkv
