// shkv_host.cu -- the C ABI of libshkv: argument checks, work planning and
// kernel launches.  Declarations and their contracts are in include/shkv.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <mutex>
#include <new>
#include <vector>

#include "shkv.h"
#include "shkv_device.cuh"
#include "prefill.cuh"
#include "tails.cuh"

namespace shkv {
cudaError_t launch_decode(int D, int NT, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          const DecodeParams &p, uint32_t smem, cudaStream_t stream);
cudaError_t launch_decode_umma(const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p, uint32_t smem,
                               cudaStream_t stream);
int umma_stages(int rows);
uint32_t umma_smem_bytes(int rows, int stages);
cudaError_t launch_append(const AppendParams &p, int num_sms, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint32_t *err, cudaStream_t stream);
cudaError_t launch_tails_units(const TailsUnitParams &p, cudaStream_t stream);
int prefill_tiles_per_cta();
uint32_t prefill_smem_bytes();
cudaError_t launch_prefill_umma(const CUtensorMap &tmK, const CUtensorMap &tmV, const PrefillParams &p, uint32_t smem,
                                int grid, cudaStream_t stream);
cudaError_t launch_merge(int n_splits, int batch, int rows, int head_dim, const float *o_part,
                         const float *lse_part, __nv_bfloat16 *out, float *lse_out, cudaStream_t stream);
}  // namespace shkv

using namespace shkv;

struct shkv_pool {
    shkv_pool_config cfg;
    int device;
    int num_sms;
    CUtensorMap tm_k;      // 3-D maps: whole row-blocks (mma.sync consumer)
    CUtensorMap tm_v;
    CUtensorMap tm_k2;     // 2-D maps: one 64-column half of a page (tcgen05 consumer)
    CUtensorMap tm_v2;
    std::vector<int32_t> lens;   // host copy of seq_lens
    bool tails_view = false;     // a per-decoder tail table over another pool's pages: empty lengths allowed
    int32_t consumer = SHKV_CONSUMER_AUTO;   // decode consumer the caller asked for
};

// Per-decoder unique tails: a view pool over the parent's pages whose
// "requests" are the (request, decoder) pairs, b * n_models + m.
struct shkv_tails {
    shkv_pool *parent;
    shkv_pool *view;
    int32_t max_batch, n_models, max_tail_pages;
};

namespace {

// Smallest number of chunks a CTA is given before the grid shrinks.
constexpr int64_t kMinChunksPerCta = 8;

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 3-D view of a [num_pages, Hkv, P, D] bf16 pool: dim0 = 64 columns
// (128 bytes, the swizzle span), dim1 = rows (num_pages*Hkv*P, stride D*2
// bytes), dim2 = D/64 column halves (stride 128 bytes).  One box
// {64, min(P, kStageTokens), D/64} with 128-byte swizzle is a whole row-block
// of one head's page -- 4 or 8 KiB in a single copy -- laid out in shared
// memory as [half][row][64 columns].
bool make_pool_map(CUtensorMap *tm, void *base, const shkv_pool_config &c)
{
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc)
        return false;
    const int halves = c.head_dim / 64;
    cuuint64_t dims[3] = {64u, (cuuint64_t)c.num_pages * c.num_kv_heads * c.page_size, (cuuint64_t)halves};
    cuuint64_t strides[2] = {(cuuint64_t)c.head_dim * 2, 128u};
    cuuint32_t box[3] = {64u, (cuuint32_t)(c.page_size < kStageTokens ? c.page_size : kStageTokens),
                         (cuuint32_t)halves};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D view of the same pool: dim0 = D columns, dim1 = rows.  One box
// {64, P} with 128-byte swizzle is one column half of one head's page,
// landing as [row][64 columns] so that consecutive pages of a stage stack
// into one 128-row operand per half.
bool make_pool_map_2d(CUtensorMap *tm, void *base, const shkv_pool_config &c)
{
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)c.head_dim, (cuuint64_t)c.num_pages * c.num_kv_heads * c.page_size};
    cuuint64_t strides[1] = {(cuuint64_t)c.head_dim * 2};
    cuuint32_t box[2] = {64u, (cuuint32_t)c.page_size};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// What a CTA's range costs the consumer that runs it, in tokens of one KV
// head streamed (a token is a row of K and a row of V, 4 * head_dim bytes).
// A range holds pieces of (request, head) units; a piece costs
//   its stages, whole: tokens rounded up to the ring's stage (the stage grid
//          starts at the piece's first page);
//   seg    the segment's query load, row sums, log-sum-exp and output write;
//   first  if it starts inside its unit (an opening split piece);
//   last   if it ends inside its unit (a closing split piece: its partial,
//          arrival and, as the last arriver, the merge, at the end of the
//          CTA's range where nothing hides them).
struct PlanCosts {
    int64_t stage, seg, first, last;
};

// tcgen05 consumer: the segment epilogue and the split merge handle one
// output row per stacked query row, so those costs grow with the rows; per
// row, in tokens: segment 12, opening piece 5, closing piece 28 (fitted to
// per-CTA exit times on GB300 at 16 rows and 16-token pages, then swept:
// closing piece 11.5 / 20 / 28 per row, opening 5 / 8 / 12, and all three
// at 0.5x and 1.5x).  mma.sync consumer: SHKV_SEGMENT_COST_CHUNKS pages a
// piece, nothing for a split (charging splits measured slower).
#ifndef SHKV_PLAN_SEG_X2
#define SHKV_PLAN_SEG_X2 24      // twice the tokens per row: segment
#endif
#ifndef SHKV_PLAN_FIRST_X2
#define SHKV_PLAN_FIRST_X2 10    // opening split piece
#endif
#ifndef SHKV_PLAN_LAST_X2
#define SHKV_PLAN_LAST_X2 56     // closing split piece
#endif
// At 16 rows the K half of a slot is refilled right after QK, so the next
// segment streams during a segment's epilogue: cheaper pieces (refitted on
// that kernel's exit times: 7, 4 and 23 tokens a row; swept against 12/5/28,
// 6/3/20, 8/4/28 and 5/4/23).
#ifndef SHKV_PLAN16_SEG_X2
#define SHKV_PLAN16_SEG_X2 14
#endif
#ifndef SHKV_PLAN16_FIRST_X2
#define SHKV_PLAN16_FIRST_X2 8
#endif
#ifndef SHKV_PLAN16_LAST_X2
#define SHKV_PLAN16_LAST_X2 46
#endif
PlanCosts plan_costs(bool umma, int32_t page_size, int32_t rows)
{
    if (umma && rows <= 16) {
        const int64_t r = rows;
        return {128, SHKV_PLAN16_SEG_X2 * r / 2, SHKV_PLAN16_FIRST_X2 * r / 2, SHKV_PLAN16_LAST_X2 * r / 2};
    }
    if (umma) {
        const int64_t r = rows;
        return {128, SHKV_PLAN_SEG_X2 * r / 2, SHKV_PLAN_FIRST_X2 * r / 2, SHKV_PLAN_LAST_X2 * r / 2};
    }
#ifndef SHKV_PLAN_MMA_FIRST
#define SHKV_PLAN_MMA_FIRST 0    // pages: opening split piece
#endif
#ifndef SHKV_PLAN_MMA_LAST
#define SHKV_PLAN_MMA_LAST 0     // pages: closing split piece
#endif
    return {page_size < kStageTokens ? page_size : kStageTokens, (int64_t)kSegmentCostChunks * page_size,
            (int64_t)SHKV_PLAN_MMA_FIRST * page_size, (int64_t)SHKV_PLAN_MMA_LAST * page_size};
}

// The split plan, shared by the plan query and the decode launch so both
// describe the same work division.  Chunks are (request, head, page) triples
// in request-major order; W = Hkv * sum_b ceil(L_b / P).  The chunk sequence
// is cut into at most `num_ctas` contiguous ranges so that the costliest
// range (under `k`) is as cheap as the greedy fill below can make it: for a
// bound B, each CTA takes whole units while it stays within B, then as many
// whole stages of the next unit as fit with that piece's closing cost; the
// smallest B for which the fill needs no more than num_ctas CTAs is found by
// bisection (it lies within one unit's fixed costs and a stage of the mean).
// Every range owns at least one chunk; fewer than num_ctas ranges can
// result, and num_ctas is then lowered to match.
//   prefix     [batch + 1] pages before each request
//   last_fill  [batch] tokens in each request's last page (nullable)
//   cuts       [num_ctas + 1] first chunk of each CTA, cuts[num_ctas] = W
shkv_status build_plan_uncached(int32_t batch, const int32_t *lens, int32_t page_size, int32_t hkv,
                                int32_t max_ctas, const PlanCosts &k, int32_t *prefix, uint8_t *last_fill,
                                int32_t *cuts, int64_t *total_chunks, int32_t *num_ctas, bool allow_empty)
{
    if (batch < 1 || batch > SHKV_MAX_BATCH || !lens || page_size <= 0 || page_size > 255 || hkv <= 0 ||
        max_ctas <= 0)
        return SHKV_ERR_INVALID_ARG;
    prefix[0] = 0;
    for (int b = 0; b < batch; ++b) {
        if (lens[b] < (allow_empty ? 0 : 1))
            return SHKV_ERR_INVALID_ARG;
        const int64_t pages = ceil_div(lens[b], page_size);
        const int64_t next = (int64_t)prefix[b] + pages;
        if (next * hkv > INT32_MAX)
            return SHKV_ERR_UNSUPPORTED;
        prefix[b + 1] = (int32_t)next;
        if (last_fill)
            last_fill[b] = (uint8_t)(pages > 0 ? lens[b] - (pages - 1) * page_size : 0);
    }
    const int64_t W = (int64_t)hkv * prefix[batch];
    int64_t C = ceil_div(W, kMinChunksPerCta);
    if (C > max_ctas)
        C = max_ctas;
    if (C > kMaxCtas)
        C = kMaxCtas;
    if (C < 1)
        C = 1;
    cuts[0] = 0;
    *total_chunks = W;
    if (W == 0) {
        for (int64_t i = 1; i <= C; ++i)
            cuts[i] = 0;
        *num_ctas = (int32_t)C;
        return SHKV_OK;
    }

    const int64_t P = page_size;
    const int64_t rb = k.stage > P ? k.stage / P : 1;           // pages a stage step covers
    const int64_t step = ceil_div(rb * P, k.stage) * k.stage;    // tokens a step costs
    auto stages = [&](int64_t pages) { return ceil_div(pages * P, k.stage) * k.stage; };
    // A unit's rest after s pages, s a whole number of steps: where pages and
    // stages nest, its stages are the unit's less the s pages.
    const bool nested = k.stage % P == 0 || P % k.stage == 0;

    // Greedy fill under bound B: the number of ranges it makes (C + 1 once it
    // needs more than C); with `out`, the cuts as well.  A request's hkv
    // units cost the same, so whole ones are taken in one step.
    std::vector<int64_t> unit_cost((size_t)batch);
    int64_t whole = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t pg = prefix[b + 1] - prefix[b];
        unit_cost[b] = pg > 0 ? k.seg + stages(pg) : 0;
        whole += hkv * unit_cost[b];
    }
    auto fill = [&](int64_t B, int32_t *out) -> int64_t {
        int64_t c = 0, acc = 0;                // current range and its cost so far
        for (int b = 0; b < batch; ++b) {
            const int64_t uc = unit_cost[b];
            if (uc == 0)
                continue;                      // an empty request owns no chunks and costs nothing
            if (acc + hkv * uc <= B) {         // the whole request fits
                acc += hkv * uc;
                continue;
            }
            const int64_t pg = prefix[b + 1] - prefix[b];
            int64_t g = 0, s = 0;              // unit of the request; its pages already given out
            while (g < hkv) {
                if (s == 0) {
                    while (g < hkv && acc + uc <= B) {
                        acc += uc;
                        ++g;
                    }
                    if (g == hkv)
                        break;
                }
                const int64_t open = k.seg + (s > 0 ? k.first : 0);
                const int64_t rest = nested ? uc - k.seg - s * P : stages(pg - s);
                if (acc + open + rest <= B) {  // the rest of a split unit
                    acc += open + rest;
                    s = 0;
                    ++g;
                    continue;
                }
                const int64_t room = B - acc - open - k.last;
                int64_t m = room > 0 ? room / step : 0;    // whole steps that fit
                const int64_t max_m = (pg - s - 1) / rb;   // leave a page for the rest
                if (m > max_m)
                    m = max_m;
                if (m == 0 && acc == 0)
                    return C + 1;              // not even one step fits an empty range
                if (++c >= C)
                    return C + 1;
                if (out)
                    out[c] = (int32_t)(hkv * prefix[b] + g * pg + s + m * rb);
                s += m * rb;
                acc = 0;
            }
        }
        return c + 1;
    };
    // The bound lies within a step and a split's fixed costs above the mean;
    // it is found to within 1/2048 of the mean (at least 16 tokens).
    const int64_t fixed_max = k.seg + k.first + k.last + step;
    const int64_t tol = std::max<int64_t>(16, whole / C / 2048);
    int64_t lo = ceil_div(whole, C) - 1;       // infeasible below the mean
    int64_t hi = ceil_div(whole, C) + fixed_max;
    while (fill(hi, nullptr) > C)
        hi += hi - lo;
    while (hi - lo > tol) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (fill(mid, nullptr) <= C)
            hi = mid;
        else
            lo = mid;
    }
    // Cuts strictly increase: a range that opens inside a unit takes at least
    // one step of it, and a cut at a unit's start closes a range that holds work.
    const int64_t used = fill(hi, cuts);
    cuts[used] = (int32_t)W;
    *num_ctas = (int32_t)used;
    return SHKV_OK;
}

// build_plan_uncached behind a one-entry cache per host thread: a call that
// repeats the previous call's inputs exactly (every layer of a model decodes
// the same lengths in a step) copies its plan instead of making it again.
shkv_status build_plan(int32_t batch, const int32_t *lens, int32_t page_size, int32_t hkv, int32_t max_ctas,
                       const PlanCosts &k, int32_t *prefix, uint8_t *last_fill, int32_t *cuts,
                       int64_t *total_chunks, int32_t *num_ctas, bool allow_empty = false)
{
    struct Entry {
        bool valid = false, allow_empty = false;
        int32_t batch = 0, page_size = 0, hkv = 0, max_ctas = 0, num_ctas = 0;
        int64_t stage = 0, seg = 0, first = 0, last = 0, total = 0;
        std::vector<int32_t> lens, prefix, cuts;
        std::vector<uint8_t> last_fill;
    };
    thread_local Entry e;
    if (e.valid && lens && batch == e.batch && page_size == e.page_size && hkv == e.hkv &&
        max_ctas == e.max_ctas && allow_empty == e.allow_empty && k.stage == e.stage && k.seg == e.seg &&
        k.first == e.first && k.last == e.last && memcmp(lens, e.lens.data(), sizeof(int32_t) * batch) == 0) {
        memcpy(prefix, e.prefix.data(), sizeof(int32_t) * (batch + 1));
        if (last_fill)
            memcpy(last_fill, e.last_fill.data(), batch);
        memcpy(cuts, e.cuts.data(), sizeof(int32_t) * (e.num_ctas + 1));
        *total_chunks = e.total;
        *num_ctas = e.num_ctas;
        return SHKV_OK;
    }
    e.valid = false;
    if (batch >= 1 && batch <= SHKV_MAX_BATCH)
        e.last_fill.resize((size_t)batch);
    const shkv_status st = build_plan_uncached(batch, lens, page_size, hkv, max_ctas, k, prefix,
                                               batch >= 1 && batch <= SHKV_MAX_BATCH ? e.last_fill.data() : nullptr,
                                               cuts, total_chunks, num_ctas, allow_empty);
    if (st != SHKV_OK)
        return st;
    if (last_fill)
        memcpy(last_fill, e.last_fill.data(), batch);
    e.lens.assign(lens, lens + batch);
    e.prefix.assign(prefix, prefix + batch + 1);
    e.cuts.assign(cuts, cuts + *num_ctas + 1);
    e.batch = batch;
    e.page_size = page_size;
    e.hkv = hkv;
    e.max_ctas = max_ctas;
    e.allow_empty = allow_empty;
    e.stage = k.stage;
    e.seg = k.seg;
    e.first = k.first;
    e.last = k.last;
    e.total = *total_chunks;
    e.num_ctas = *num_ctas;
    e.valid = true;
    return SHKV_OK;
}

// A decode's workspace: the arrival counters (one per (request, head) unit)
// in a region of fixed size at its front, then the split pieces' lse and
// partials.  The counters of every call, whatever its shape, live in that
// region and nothing else is ever written there, so a workspace whose region
// starts zeroed stays zeroed between calls (the last arriver of each unit
// clears its counter) when consecutive calls change batch or shape.
constexpr size_t kCountRegion = SHKV_COUNT_REGION_BYTES;

// Bytes of the counter region: the fixed region, or (compact) only this
// call's counters, for a scratch whose counters every call clears first.
size_t count_region_bytes(int32_t batch, int32_t hkv, bool compact)
{
    return compact ? align_up((uint32_t)(batch * hkv * 4), 256) : kCountRegion;
}

size_t workspace_bytes_for(int32_t batch, int32_t hkv, int32_t rows, int32_t head_dim, int32_t num_sms,
                           bool compact = false)
{
    const size_t lse = align_up((uint32_t)(2 * num_sms * rows * 4), 256);
    const size_t part = (size_t)2 * num_sms * rows * head_dim * 4;
    return count_region_bytes(batch, hkv, compact) + lse + part;
}

shkv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SHKV_OK : SHKV_ERR_CUDA; }

// Device bytes [lo, hi).
struct Span {
    uintptr_t lo, hi;
};

Span span_of(const void *p, size_t bytes)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, p ? a + bytes : a};
}

// The device bytes that the library's last kernel-launching call on each
// stream reads or writes (its workspace bytes, queries, outputs, tables).
// Every library kernel lets the next kernel of its stream start once it has
// passed its own wait, so when a tails call's layout kernel starts, that
// call's last kernel may still run while everything before it has
// completed.  The layout kernel writes its tables before waiting only at an
// offset of its workspace whose bytes miss all of these spans, whatever
// pointer the earlier call used for them; when none fits, or the stream has
// no record, it waits for the previous kernel first.  A small table keyed by
// stream, least recently used out after 64 others (a stream whose record
// was dropped just waits).
struct StreamUse {
    static constexpr int kMaxSpans = 8;
    struct Entry {
        const void *stream;
        uint64_t used;
        int n;
        Span s[kMaxSpans];
    };
    std::mutex mu;
    std::vector<Entry> entries;
    uint64_t clock = 0;

    // Offset of `bytes` of tables in workspace `ws` of `limit` bytes, at or
    // after `d` (this call's decode part), for a call on `stream`.
    size_t place(const void *stream, const uint8_t *ws, size_t d, size_t bytes, size_t limit, bool *wait_first)
    {
        std::lock_guard<std::mutex> g(mu);
        *wait_first = true;
        const uintptr_t base = reinterpret_cast<uintptr_t>(ws);
        for (const Entry &e : entries) {
            if (e.stream != stream)
                continue;
            size_t cands[kMaxSpans + 2];
            int nc = 0;
            cands[nc++] = d;
            for (int i = 0; i < e.n; ++i)
                if (e.s[i].hi > base + d && e.s[i].hi - base <= limit)
                    cands[nc++] = (e.s[i].hi - base + 255) / 256 * 256;
            if (limit >= bytes)
                cands[nc++] = (limit - bytes) / 256 * 256;
            size_t best = limit;                 // the lowest candidate that fits and is clear
            for (int ci = 0; ci < nc; ++ci) {
                const size_t c = cands[ci];
                if (c < d || c + bytes > limit || c >= best)
                    continue;
                bool clear = true;
                for (int i = 0; i < e.n && clear; ++i)
                    clear = e.s[i].hi <= base + c || e.s[i].lo >= base + c + bytes;
                if (clear)
                    best = c;
            }
            if (best == limit)
                return d;
            *wait_first = false;
            return best;
        }
        return d;
    }
    // After a call on `stream` enqueued at least one kernel: the spans it
    // touches (empty spans are skipped).
    void record(const void *stream, std::initializer_list<Span> spans)
    {
        std::lock_guard<std::mutex> g(mu);
        Entry rec{stream, ++clock, 0, {}};
        for (const Span &s : spans)
            if (s.hi > s.lo && rec.n < kMaxSpans)
                rec.s[rec.n++] = s;
        for (Entry &e : entries)
            if (e.stream == stream) {
                e = rec;
                return;
            }
        if (entries.size() >= 64) {
            auto lru = std::min_element(entries.begin(), entries.end(),
                                        [](const Entry &x, const Entry &y) { return x.used < y.used; });
            entries.erase(lru);
        }
        entries.push_back(rec);
    }
};
StreamUse g_stream_use;

// Launch shape of the decode kernel for R stacked rows per KV head.
struct DecodeShape {
    int nt, nrg, wt, rpad;
};

DecodeShape decode_shape(int rows)
{
    DecodeShape s;
    if (rows <= 8) {
        s.nt = 1;
        s.nrg = 1;
        s.wt = SHKV_WT_NT1;
    } else if (rows <= 16 || !SHKV_R_ABOVE16_NT1) {
        s.nt = 2;
        s.nrg = (rows + 15) / 16;
        s.wt = kWtOfNrg[s.nrg];
    } else {
        s.nt = 1;
        s.nrg = (rows + 7) / 8;
        s.wt = kNt1MultiWarps / s.nrg > 0 ? kNt1MultiWarps / s.nrg : 1;
        if (s.wt > kWtMax)
            s.wt = kWtMax;
    }
    s.rpad = s.nrg * 8 * s.nt;
    return s;
}

// Which consumer runs for R stacked rows of head dim D: the one the pool
// names (shkv_pool_set_decode_consumer), else the automatic policy.  The
// tcgen05 consumer covers D = 128 and R <= 64 only; outside that the
// mma.sync consumer runs whatever the pool names.
bool use_umma_consumer(int rows, int head_dim, int32_t choice)
{
    if (head_dim != 128 || rows > kUmmaMaxRows || umma_stages(rows) == 0)
        return false;
    if (choice == SHKV_CONSUMER_TCGEN05)
        return true;
    if (choice == SHKV_CONSUMER_MMA_SYNC)
        return false;
    return rows >= kUmmaMinRows;
}

}  // namespace

extern "C" {

const char *shkv_status_string(shkv_status s)
{
    switch (s) {
    case SHKV_OK:
        return "ok";
    case SHKV_ERR_INVALID_ARG:
        return "invalid argument";
    case SHKV_ERR_CAPACITY:
        return "sequence exceeds the pool's per-request capacity";
    case SHKV_ERR_UNSUPPORTED:
        return "unsupported shape or configuration";
    case SHKV_ERR_CUDA:
        return "CUDA runtime error";
    case SHKV_ERR_DEVICE:
        return "device error bits set";
    }
    return "unknown status";
}

shkv_status shkv_pool_create(const shkv_pool_config *cfg, shkv_pool **out)
{
    if (!cfg || !out)
        return SHKV_ERR_INVALID_ARG;
    *out = nullptr;
    const shkv_pool_config &c = *cfg;
    if (c.num_pages <= 0 || c.num_kv_heads <= 0 || c.max_batch <= 0 || c.max_pages_per_seq <= 0 ||
        !c.k_pages || !c.v_pages || !c.block_table || !c.seq_lens || !c.error_word)
        return SHKV_ERR_INVALID_ARG;
    if (!aligned16(c.k_pages) || !aligned16(c.v_pages) || ((uintptr_t)c.block_table & 3u) ||
        ((uintptr_t)c.seq_lens & 3u) || ((uintptr_t)c.error_word & 3u))
        return SHKV_ERR_INVALID_ARG;
    if ((c.page_size != 16 && c.page_size != 32) || (c.head_dim != 64 && c.head_dim != 128))
        return SHKV_ERR_UNSUPPORTED;
    if ((int64_t)c.num_pages * c.num_kv_heads * c.page_size > INT32_MAX ||
        (int64_t)c.max_pages_per_seq * c.page_size > INT32_MAX)
        return SHKV_ERR_UNSUPPORTED;
    if (c.initial_seq_lens)
        for (int b = 0; b < c.max_batch; ++b)
            if (c.initial_seq_lens[b] < 0 || (int64_t)c.initial_seq_lens[b] > (int64_t)c.max_pages_per_seq * c.page_size)
                return SHKV_ERR_CAPACITY;

    shkv_pool *pool = new (std::nothrow) shkv_pool();
    if (!pool)
        return SHKV_ERR_INVALID_ARG;
    pool->cfg = c;
    pool->cfg.initial_seq_lens = nullptr;
    pool->lens.assign(c.max_batch, 0);
    if (c.initial_seq_lens)
        memcpy(pool->lens.data(), c.initial_seq_lens, sizeof(int32_t) * c.max_batch);
    if (cudaGetDevice(&pool->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&pool->num_sms, cudaDevAttrMultiProcessorCount, pool->device) != cudaSuccess) {
        delete pool;
        return SHKV_ERR_CUDA;
    }
    if (!make_pool_map(&pool->tm_k, c.k_pages, c) || !make_pool_map(&pool->tm_v, c.v_pages, c) ||
        !make_pool_map_2d(&pool->tm_k2, c.k_pages, c) || !make_pool_map_2d(&pool->tm_v2, c.v_pages, c)) {
        delete pool;
        return SHKV_ERR_CUDA;
    }
    if (cudaMemcpy(c.seq_lens, pool->lens.data(), sizeof(int32_t) * c.max_batch, cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemset(c.error_word, 0, sizeof(uint32_t)) != cudaSuccess) {
        delete pool;
        return SHKV_ERR_CUDA;
    }
    *out = pool;
    return SHKV_OK;
}

shkv_status shkv_pool_destroy(shkv_pool *pool)
{
    if (!pool)
        return SHKV_ERR_INVALID_ARG;
    delete pool;
    return SHKV_OK;
}

shkv_status shkv_pool_set_seq_lens(shkv_pool *pool, int32_t batch, const int32_t *lens, void *stream)
{
    if (!pool || !lens || batch < 0 || batch > pool->cfg.max_batch)
        return SHKV_ERR_INVALID_ARG;
    const int64_t cap = (int64_t)pool->cfg.max_pages_per_seq * pool->cfg.page_size;
    for (int b = 0; b < batch; ++b)
        if (lens[b] < 0 || lens[b] > cap)
            return SHKV_ERR_CAPACITY;
    if (batch == 0)
        return SHKV_OK;
    memcpy(pool->lens.data(), lens, sizeof(int32_t) * batch);
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(pool->cfg.seq_lens, pool->lens.data(), sizeof(int32_t) * batch,
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(st);
    return cuda_status(e);
}

shkv_status shkv_pool_get_seq_lens(const shkv_pool *pool, int32_t batch, int32_t *lens)
{
    if (!pool || !lens || batch < 0 || batch > pool->cfg.max_batch)
        return SHKV_ERR_INVALID_ARG;
    memcpy(lens, pool->lens.data(), sizeof(int32_t) * batch);
    return SHKV_OK;
}

shkv_status shkv_append_kv(shkv_pool *pool, int32_t batch, int32_t n_new_tokens, const void *k_new,
                           const void *v_new, void *stream)
{
    if (!pool || batch < 0 || batch > pool->cfg.max_batch || batch > SHKV_MAX_BATCH || n_new_tokens < 0)
        return SHKV_ERR_INVALID_ARG;
    if (batch == 0 || n_new_tokens == 0)
        return SHKV_OK;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
        return SHKV_ERR_INVALID_ARG;
    const shkv_pool_config &c = pool->cfg;
    const int64_t cap = (int64_t)c.max_pages_per_seq * c.page_size;
    for (int b = 0; b < batch; ++b)
        if ((int64_t)pool->lens[b] + n_new_tokens > cap)
            return SHKV_ERR_CAPACITY;
    AppendParams p;
    memset(&p, 0, sizeof p);
    p.k_new = reinterpret_cast<const uint4 *>(k_new);
    p.v_new = reinterpret_cast<const uint4 *>(v_new);
    p.k_pages = reinterpret_cast<uint4 *>(c.k_pages);
    p.v_pages = reinterpret_cast<uint4 *>(c.v_pages);
    p.block_table = c.block_table;
    p.seq_lens = c.seq_lens;
    p.err = c.error_word;
    p.batch = batch;
    p.n_new = n_new_tokens;
    p.hkv = c.num_kv_heads;
    p.head_vecs = c.head_dim / 8;
    p.page_size = c.page_size;
    p.max_pages = c.max_pages_per_seq;
    p.num_pages = c.num_pages;
    for (int b = 0; b < batch; ++b)
        p.old_len[b] = pool->lens[b];
    cudaError_t e = launch_append(p, pool->num_sms, (cudaStream_t)stream);
    if (e != cudaSuccess)
        return SHKV_ERR_CUDA;
    const size_t new_bytes = (size_t)batch * n_new_tokens * c.num_kv_heads * c.head_dim * 2;
    g_stream_use.record(stream, {span_of(k_new, new_bytes), span_of(v_new, new_bytes)});
    for (int b = 0; b < batch; ++b)
        pool->lens[b] += n_new_tokens;
    return SHKV_OK;
}

shkv_status shkv_decode_workspace_size(const shkv_pool *pool, int32_t batch, int32_t n_models,
                                       int32_t hq_per_model, size_t *bytes)
{
    if (!pool || !bytes || batch < 1 || n_models < 1 || hq_per_model < 1)
        return SHKV_ERR_INVALID_ARG;
    const int hkv = pool->cfg.num_kv_heads;
    if (hq_per_model % hkv)
        return SHKV_ERR_UNSUPPORTED;
    const int rows = n_models * (hq_per_model / hkv);
    *bytes = workspace_bytes_for(batch, hkv, rows, pool->cfg.head_dim, pool->num_sms);
    return SHKV_OK;
}

}  // extern "C"

namespace {

// Units of a decode with per-decoder tails in one pass: the unit table and
// page info built on the device, their row stride, and each request's unit
// length in tokens (whole pages), which the split plan is built from.

struct FusedUnits {
    const int32_t *table;
    const uint32_t *info;
    int32_t stride;
    const int32_t *unit_tokens;
};

// One decode launch: final rows to out (bf16).  Launches nothing when the pool has
// no chunks (every length zero, possible only for a tail view).  With fu,
// request b's unit is fu's row b instead of the pool's block table.  With
// clear_counters, once every check has passed, the workspace's arrival
// counters are zeroed on the stream before the launch (for a workspace whose
// previous contents are unknown).  before_launch, if given, is called once
// every check has passed, right before the decode kernel is enqueued (the
// tails path enqueues its unit kernel there); its error aborts the call.
shkv_status decode_impl(shkv_pool *pool, int32_t batch, int32_t n_models, int32_t hq_per_model, const void *q,
                        float scale, void *out, float *lse_out, void *workspace,
                        size_t workspace_bytes, void *stream, const FusedUnits *fu = nullptr,
                        bool clear_counters = false, const std::function<cudaError_t()> *before_launch = nullptr,
                        Span tables = {0, 0})
{
    if (!pool || !q || !out || !workspace || batch < 1 || n_models < 1 ||
        hq_per_model < 1)
        return SHKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) ||
        ((uintptr_t)lse_out & 3u))
        return SHKV_ERR_INVALID_ARG;
    if (!isfinite(scale))
        return SHKV_ERR_INVALID_ARG;
    const shkv_pool_config &c = pool->cfg;
    if (batch > c.max_batch)
        return SHKV_ERR_INVALID_ARG;
    if (batch > SHKV_MAX_BATCH || hq_per_model % c.num_kv_heads)
        return SHKV_ERR_UNSUPPORTED;
    const int group = hq_per_model / c.num_kv_heads;
    const int rows = n_models * group;
    if (rows > 64)
        return SHKV_ERR_UNSUPPORTED;
    if ((int64_t)batch * c.num_kv_heads * 4 > (int64_t)kCountRegion)
        return SHKV_ERR_UNSUPPORTED;
    if (workspace_bytes < workspace_bytes_for(batch, c.num_kv_heads, rows, c.head_dim, pool->num_sms, clear_counters))
        return SHKV_ERR_INVALID_ARG;

    const bool use_umma = use_umma_consumer(rows, c.head_dim, pool->consumer);
    DecodeParams p;
    memset(&p, 0, sizeof p);
    shkv_status st = build_plan(batch, fu ? fu->unit_tokens : pool->lens.data(), c.page_size, c.num_kv_heads,
                                pool->num_sms, plan_costs(use_umma, c.page_size, rows), p.page_prefix, p.last_fill,
                                p.cta_cut, &p.total_chunks, &p.num_ctas, pool->tails_view);
    if (st != SHKV_OK)
        return st;
    if (p.total_chunks == 0)
        return SHKV_OK;

    const DecodeShape sh = decode_shape(rows);
    const int ncw = sh.nrg * sh.wt;
    const int nreg = (c.head_dim / 16) * sh.nt * 4;
    const DecodeSmem probe = decode_smem_layout(c.head_dim, 8 * sh.nt, nreg, ncw, sh.rpad, 0);
    int stages = (int)((kSmemLimit - (int64_t)probe.total - 64) / (probe.stage_bytes + 20));
    if (stages > kMaxStages)
        stages = kMaxStages;
    // Consumer warp w of a row group takes stages k = w (mod wt), so with a
    // ring of a multiple of wt slots the previous occupant of its next slot
    // is its own, already consumed, stage: its parity wait can never see an
    // older phase of the slot.
    stages -= stages % sh.wt;
    uint32_t smem_bytes = 0;
    if (use_umma) {
        // one consumer (the MMA issuer) takes every stage in order: any ring size
        stages = umma_stages(rows);
        smem_bytes = umma_smem_bytes(rows, stages);
    } else {
        if (stages < 2 || stages < sh.wt)
            return SHKV_ERR_UNSUPPORTED;
        const DecodeSmem lay = decode_smem_layout(c.head_dim, 8 * sh.nt, nreg, ncw, sh.rpad, stages);
        if (lay.total > (uint32_t)kSmemLimit)
            return SHKV_ERR_UNSUPPORTED;
        smem_bytes = lay.total;
    }

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t count_bytes = align_up((uint32_t)(batch * c.num_kv_heads * 4), 256);   // in use by this call
    const size_t lse_bytes = align_up((uint32_t)(2 * pool->num_sms * rows * 4), 256);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.lse_out = lse_out;
    p.block_table = fu ? fu->table : c.block_table;
    p.page_info = fu ? fu->info : nullptr;
    p.fused = fu ? 1 : 0;
    p.seq_lens = c.seq_lens;
    p.err = c.error_word;
    p.ws_count = reinterpret_cast<uint32_t *>(ws);
    const size_t count_region = count_region_bytes(batch, c.num_kv_heads, clear_counters);
    p.ws_lse = reinterpret_cast<float *>(ws + count_region);
    p.ws_part = reinterpret_cast<float *>(ws + count_region + lse_bytes);
    p.batch = batch;
    p.n_models = n_models;
    p.hq = hq_per_model;
    p.hkv = c.num_kv_heads;
    p.group = group;
    p.rows = rows;
    p.nrg = sh.nrg;
    p.wt = sh.wt;
    p.rpad = sh.rpad;
    p.stages = stages;
    p.page_size = c.page_size;
    p.box_rows = c.page_size < kStageTokens ? c.page_size : kStageTokens;
    p.max_pages = fu ? fu->stride : c.max_pages_per_seq;
    p.num_pages = c.num_pages;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    // tcgen05 consumer: 16-token pages make 32 copies a stage, issued by two
    // warps; the 16 copies of 32-token pages measured faster from one warp
    p.split_producers = c.page_size < 32 ? 1 : 0;
    if (clear_counters && cudaMemsetAsync(p.ws_count, 0, count_bytes, (cudaStream_t)stream) != cudaSuccess)
        return SHKV_ERR_CUDA;
    if (before_launch && (*before_launch)() != cudaSuccess)
        return SHKV_ERR_CUDA;
    cudaError_t e = use_umma ? launch_decode_umma(pool->tm_k2, pool->tm_v2, p, smem_bytes, (cudaStream_t)stream)
                             : launch_decode(c.head_dim, sh.nt, pool->tm_k, pool->tm_v, p, smem_bytes,
                                             (cudaStream_t)stream);
    // what this call's kernels touch, for a tails call after it on the stream
    // (recorded also when the decode launch failed after the unit kernel's)
    const size_t qrows = (size_t)batch * n_models * hq_per_model;
    g_stream_use.record(stream, {span_of(workspace, workspace_bytes_for(batch, c.num_kv_heads, rows, c.head_dim,
                                                                        pool->num_sms, clear_counters)),
                                 span_of(q, qrows * c.head_dim * 2), span_of(out, qrows * c.head_dim * 2),
                                 span_of(lse_out, qrows * 4), tables});
    return cuda_status(e);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Workspace of a decode with tails: the decode's own, then the unit table
// and page info [B, stride] with stride = max_pages_per_seq + N * max_tail_pages.
struct TailsWorkspace {
    size_t decode, table, stride, total;
};

TailsWorkspace tails_workspace(const shkv_pool *pool, const shkv_tails *tails, int32_t batch, int32_t group)
{
    const shkv_pool_config &c = pool->cfg;
    TailsWorkspace w;
    w.decode = align256(workspace_bytes_for(batch, c.num_kv_heads, tails->n_models * group, c.head_dim,
                                            pool->num_sms));
    w.stride = (size_t)c.max_pages_per_seq + (size_t)tails->n_models * tails->max_tail_pages;
    w.table = align256((size_t)batch * w.stride * 4);
    w.total = w.decode + 4 * w.table;          // room for two positions of (unit table, page words)
    return w;
}


}  // namespace

extern "C" {

shkv_status shkv_decode_attention(shkv_pool *pool, int32_t batch, int32_t n_models, int32_t hq_per_model,
                                  const void *q, float scale, void *out, float *lse_out, void *workspace,
                                  size_t workspace_bytes, void *stream)
{
    if (!out)
        return SHKV_ERR_INVALID_ARG;
    return decode_impl(pool, batch, n_models, hq_per_model, q, scale, out, lse_out, workspace, workspace_bytes,
                       stream);
}

shkv_status shkv_prefill_attention(shkv_pool *pool, int32_t batch, int32_t n_new, int32_t hq_per_model,
                                   const void *q, float scale, void *out, float *lse_out, void *stream)
{
    if (!pool || !q || !out || batch < 1 || n_new < 1 || hq_per_model < 1 || !isfinite(scale))
        return SHKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out) || ((uintptr_t)lse_out & 3u))
        return SHKV_ERR_INVALID_ARG;
    const shkv_pool_config &c = pool->cfg;
    if (batch > c.max_batch)
        return SHKV_ERR_INVALID_ARG;
    if (batch > SHKV_MAX_BATCH || hq_per_model % c.num_kv_heads || c.head_dim != 128 || pool->tails_view)
        return SHKV_ERR_UNSUPPORTED;
    const int group = hq_per_model / c.num_kv_heads;
    if (group > 128)
        return SHKV_ERR_UNSUPPORTED;
    PrefillParams p;
    memset(&p, 0, sizeof p);
    for (int b = 0; b < batch; ++b) {
        if (pool->lens[b] < n_new)
            return SHKV_ERR_INVALID_ARG;        // the new tokens must already be in the pool
        p.lens[b] = pool->lens[b];
        p.order[b] = b;
    }
    std::stable_sort(p.order, p.order + batch, [&](int32_t a, int32_t b) { return p.lens[a] > p.lens[b]; });
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.lse_out = lse_out;
    p.block_table = c.block_table;
    p.seq_lens = c.seq_lens;
    p.err = c.error_word;
    p.batch = batch;
    p.n_new = n_new;
    p.hq = hq_per_model;
    p.hkv = c.num_kv_heads;
    p.group = group;
    p.tpt = 128 / group;
    p.tiles = (n_new + p.tpt - 1) / p.tpt;
    p.page_size = c.page_size;
    p.max_pages = c.max_pages_per_seq;
    p.num_pages = c.num_pages;
    p.stages = 0;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    const int per_cta = prefill_tiles_per_cta();
    const int64_t grid = (int64_t)batch * c.num_kv_heads * ((p.tiles + per_cta - 1) / per_cta);
    if (grid > INT32_MAX)
        return SHKV_ERR_UNSUPPORTED;
    const cudaError_t e =
        launch_prefill_umma(pool->tm_k2, pool->tm_v2, p, prefill_smem_bytes(), (int)grid, (cudaStream_t)stream);
    if (e == cudaSuccess) {
        const size_t qrows = (size_t)batch * n_new * hq_per_model;
        g_stream_use.record(stream, {span_of(q, qrows * c.head_dim * 2), span_of(out, qrows * c.head_dim * 2),
                                     span_of(lse_out, qrows * 4)});
    }
    return cuda_status(e);
}

shkv_status shkv_tails_create(shkv_pool *pool, const shkv_tails_config *tc, shkv_tails **out)
{
    if (!pool || !tc || !out)
        return SHKV_ERR_INVALID_ARG;
    *out = nullptr;
    if (pool->tails_view || tc->max_batch < 1 || tc->n_models < 1 || tc->max_tail_pages < 1 || !tc->block_table ||
        !tc->tail_lens || ((uintptr_t)tc->block_table & 3u) || ((uintptr_t)tc->tail_lens & 3u))
        return SHKV_ERR_INVALID_ARG;
    if ((int64_t)tc->max_batch * tc->n_models > INT32_MAX / 2)
        return SHKV_ERR_UNSUPPORTED;
    shkv_pool_config vc = pool->cfg;
    vc.max_batch = tc->max_batch * tc->n_models;
    vc.max_pages_per_seq = tc->max_tail_pages;
    vc.block_table = tc->block_table;
    vc.seq_lens = tc->tail_lens;
    vc.initial_seq_lens = tc->initial_tail_lens;
    shkv_tails *t = new (std::nothrow) shkv_tails();
    if (!t)
        return SHKV_ERR_INVALID_ARG;
    // the view shares the parent's pages and error word; creating it writes
    // the tail lengths to the device and clears the (shared) error word
    shkv_status st = shkv_pool_create(&vc, &t->view);
    if (st != SHKV_OK) {
        delete t;
        return st;
    }
    t->view->tails_view = true;
    t->parent = pool;
    t->max_batch = tc->max_batch;
    t->n_models = tc->n_models;
    t->max_tail_pages = tc->max_tail_pages;
    *out = t;
    return SHKV_OK;
}

shkv_status shkv_tails_destroy(shkv_tails *tails)
{
    if (!tails)
        return SHKV_ERR_INVALID_ARG;
    shkv_pool_destroy(tails->view);
    delete tails;
    return SHKV_OK;
}

shkv_status shkv_tails_set_lens(shkv_tails *tails, int32_t batch, const int32_t *tail_lens, void *stream)
{
    if (!tails || batch < 0 || batch > tails->max_batch)
        return SHKV_ERR_INVALID_ARG;
    return shkv_pool_set_seq_lens(tails->view, batch * tails->n_models, tail_lens, stream);
}

shkv_status shkv_tails_get_lens(const shkv_tails *tails, int32_t batch, int32_t *tail_lens)
{
    if (!tails || batch < 0 || batch > tails->max_batch)
        return SHKV_ERR_INVALID_ARG;
    return shkv_pool_get_seq_lens(tails->view, batch * tails->n_models, tail_lens);
}

shkv_status shkv_tails_append(shkv_tails *tails, int32_t batch, int32_t n_new_tokens, const void *k_new,
                              const void *v_new, void *stream)
{
    if (!tails || batch < 1 || batch > tails->max_batch)
        return SHKV_ERR_INVALID_ARG;
    return shkv_append_kv(tails->view, batch * tails->n_models, n_new_tokens, k_new, v_new, stream);
}

shkv_status shkv_decode_tails_workspace_size(const shkv_pool *pool, const shkv_tails *tails, int32_t batch,
                                             int32_t hq_per_model, size_t *bytes)
{
    if (!pool || !tails || !bytes || tails->parent != pool || batch < 1 || hq_per_model < 1)
        return SHKV_ERR_INVALID_ARG;
    if (hq_per_model % pool->cfg.num_kv_heads)
        return SHKV_ERR_UNSUPPORTED;
    *bytes = tails_workspace(pool, tails, batch, hq_per_model / pool->cfg.num_kv_heads).total;
    return SHKV_OK;
}

shkv_status shkv_decode_attention_tails(shkv_pool *pool, shkv_tails *tails, int32_t batch, int32_t hq_per_model,
                                        const void *q, float scale, void *out, float *lse_out, void *workspace,
                                        size_t workspace_bytes, void *stream)
{
    if (!pool || !tails || tails->parent != pool || !q || !out || !workspace || batch < 1 || hq_per_model < 1)
        return SHKV_ERR_INVALID_ARG;
    if (batch > tails->max_batch || batch > pool->cfg.max_batch)
        return SHKV_ERR_INVALID_ARG;
    if (hq_per_model % pool->cfg.num_kv_heads)
        return SHKV_ERR_UNSUPPORTED;
    const int32_t N = tails->n_models;
    if ((int64_t)batch * N > SHKV_MAX_BATCH)
        return SHKV_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) || ((uintptr_t)lse_out & 3u))
        return SHKV_ERR_INVALID_ARG;
    if (N > 254 ||
        ((int64_t)pool->cfg.max_pages_per_seq + (int64_t)N * tails->max_tail_pages) * pool->cfg.page_size > INT32_MAX)
        return SHKV_ERR_UNSUPPORTED;
    const int group = hq_per_model / pool->cfg.num_kv_heads;
    const TailsWorkspace w = tails_workspace(pool, tails, batch, group);
    if (workspace_bytes < w.total)
        return SHKV_ERR_INVALID_ARG;
    // One pass: request b's unit is its shared pages then each decoder's tail
    // pages; a tail page is attended by its decoder's rows only.
    const int32_t P = pool->cfg.page_size;
    TailsUnitParams up;
    memset(&up, 0, sizeof up);
    std::vector<int32_t> unit_tokens((size_t)batch);
    for (int b = 0; b < batch; ++b) {
        const int32_t L = pool->lens[b];
        if (L < 1)
            return SHKV_ERR_INVALID_ARG;
        up.shared_len[b] = L;
        int64_t pages = (L + P - 1) / P;
        for (int m = 0; m < N; ++m) {
            const int32_t T = tails->view->lens[(size_t)b * N + m];
            up.tail_len[b * N + m] = T;
            pages += (T + P - 1) / P;
        }
        unit_tokens[b] = (int32_t)(pages * P);
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    bool wait_first = false;
    const size_t off = g_stream_use.place(stream, ws, w.decode, 2 * w.table, workspace_bytes, &wait_first);
    up.block_table = pool->cfg.block_table;
    up.tail_table = tails->view->cfg.block_table;
    up.unit_table = reinterpret_cast<int32_t *>(ws + off);
    up.unit_info = reinterpret_cast<uint32_t *>(ws + off + w.table);
    up.wait_first = wait_first ? 1 : 0;
    up.bt_stride = pool->cfg.max_pages_per_seq;
    up.tt_stride = tails->max_tail_pages;
    up.ustride = (int32_t)w.stride;
    up.batch = batch;
    up.n_models = N;
    up.page_size = P;
    // the unit kernel is enqueued right before the decode, once every check
    // of the decode has passed (never alone, so the last tables a workspace
    // recorded are the ones its last decode reads)
    const std::function<cudaError_t()> units = [&]() { return launch_tails_units(up, (cudaStream_t)stream); };
    const FusedUnits fu{up.unit_table, up.unit_info, up.ustride, unit_tokens.data()};
    return decode_impl(pool, batch, N, hq_per_model, q, scale, out, lse_out, ws, w.decode, stream, &fu, false,
                       &units, span_of(ws + off, 2 * w.table));
}

shkv_status shkv_decode_consumer(const shkv_pool *pool, int32_t n_models, int32_t hq_per_model, int32_t *consumer)
{
    if (!pool || !consumer || n_models < 1 || hq_per_model < 1)
        return SHKV_ERR_INVALID_ARG;
    if (hq_per_model % pool->cfg.num_kv_heads)
        return SHKV_ERR_UNSUPPORTED;
    const int rows = n_models * (hq_per_model / pool->cfg.num_kv_heads);
    if (rows > 64)
        return SHKV_ERR_UNSUPPORTED;
    *consumer = use_umma_consumer(rows, pool->cfg.head_dim, pool->consumer) ? SHKV_CONSUMER_TCGEN05
                                                                            : SHKV_CONSUMER_MMA_SYNC;
    return SHKV_OK;
}

shkv_status shkv_pool_set_decode_consumer(shkv_pool *pool, int32_t consumer)
{
    if (!pool || (consumer != SHKV_CONSUMER_AUTO && consumer != SHKV_CONSUMER_MMA_SYNC &&
                  consumer != SHKV_CONSUMER_TCGEN05))
        return SHKV_ERR_INVALID_ARG;
    pool->consumer = consumer;
    return SHKV_OK;
}

shkv_status shkv_splitkv_merge(int32_t n_splits, int32_t batch, int32_t rows, int32_t head_dim, const float *o_part,
                               const float *lse_part, void *out, float *lse_out, void *stream)
{
    if (n_splits < 1 || batch < 0 || rows < 0 || head_dim <= 0 || head_dim % 4 || !o_part || !lse_part || !out)
        return SHKV_ERR_INVALID_ARG;
    if (!aligned16(o_part) || ((uintptr_t)lse_part & 3u) || ((uintptr_t)out & 7u) || ((uintptr_t)lse_out & 3u))
        return SHKV_ERR_INVALID_ARG;
    cudaError_t e = launch_merge(n_splits, batch, rows, head_dim, o_part, lse_part,
                                 static_cast<__nv_bfloat16 *>(out), lse_out, (cudaStream_t)stream);
    const size_t nrow = (size_t)batch * rows;
    if (e == cudaSuccess && nrow > 0)
        g_stream_use.record(stream, {span_of(o_part, n_splits * nrow * head_dim * 4),
                                     span_of(lse_part, n_splits * nrow * 4), span_of(out, nrow * head_dim * 2),
                                     span_of(lse_out, nrow * 4)});
    return cuda_status(e);
}

shkv_status shkv_selftest_bounded_wait(shkv_pool *pool, void *stream)
{
    if (!pool)
        return SHKV_ERR_INVALID_ARG;
    return cuda_status(launch_wait_selftest(pool->cfg.error_word, (cudaStream_t)stream));
}

shkv_status shkv_check_errors(shkv_pool *pool, void *stream, uint32_t *flags)
{
    if (!pool || !flags)
        return SHKV_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    *flags = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return SHKV_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, pool->cfg.error_word, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SHKV_ERR_CUDA;
    if (v && cudaMemset(pool->cfg.error_word, 0, sizeof v) != cudaSuccess)
        return SHKV_ERR_CUDA;
    *flags = v;
    return v ? SHKV_ERR_DEVICE : SHKV_OK;
}

shkv_status shkv_plan_decode(int32_t batch, const int32_t *seq_lens, int32_t page_size, int32_t num_kv_heads,
                             int32_t n_models, int32_t hq_per_model, int32_t consumer, int32_t max_ctas,
                             int64_t *cta_begin, int32_t *num_ctas, int32_t *num_splits)
{
    if (!num_ctas || (consumer != SHKV_CONSUMER_MMA_SYNC && consumer != SHKV_CONSUMER_TCGEN05) || n_models < 1 ||
        hq_per_model < 1 || num_kv_heads < 1)
        return SHKV_ERR_INVALID_ARG;
    if (hq_per_model % num_kv_heads || n_models * (int64_t)(hq_per_model / num_kv_heads) > 64)
        return SHKV_ERR_UNSUPPORTED;
    const int32_t rows = n_models * (hq_per_model / num_kv_heads);
    std::vector<int32_t> prefix((size_t)SHKV_MAX_BATCH + 1);
    std::vector<int32_t> cuts((size_t)kMaxCtas + 1);
    int64_t W = 0;
    int32_t C = 0;
    shkv_status st = build_plan(batch, seq_lens, page_size, num_kv_heads, max_ctas,
                                plan_costs(consumer == SHKV_CONSUMER_TCGEN05, page_size, rows), prefix.data(), nullptr,
                                cuts.data(), &W, &C);
    if (st != SHKV_OK)
        return st;
    *num_ctas = C;
    if (cta_begin)
        for (int c = 0; c <= C; ++c)
            cta_begin[c] = cuts[c];
    if (num_splits) {
        // one pass over units and cuts together: with cuts[c] <= u0 < cuts[c + 1],
        // the unit [u0, u1) is split iff cuts[c + 1] < u1
        int32_t n = 0, c = 0;
        for (int b = 0; b < batch; ++b) {
            const int64_t pages = prefix[b + 1] - prefix[b];
            for (int g = 0; g < num_kv_heads && pages > 0; ++g) {
                const int64_t u0 = (int64_t)num_kv_heads * prefix[b] + g * pages;
                while (c + 1 < C && cuts[c + 1] <= u0)
                    ++c;
                if (c + 1 < C && cuts[c + 1] < u0 + pages)
                    ++n;
            }
        }
        *num_splits = n;
    }
    return SHKV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// decode without a caller workspace: static device scratch
// ---------------------------------------------------------------------------
// The split-KV scratch of shkv_decode_attention_noalloc.  Device globals are
// zero-initialised when the module loads; each call re-zeroes the arrival
// counters at its front before launching.
static __device__ __align__(256) unsigned char shkv_noalloc_scratch[SHKV_NOALLOC_SCRATCH_BYTES];

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Driver entry points reached through the runtime, so the library needs no
// libcuda at load time (as for the tensor-map encoder).
template <typename Fn>
Fn driver_fn(const char *name, int version)
{
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &ptr, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(ptr);
}

// Unique ID (within the process) of the context current on this thread, or
// 0 when none is current.  IDs are never reused, unlike context handles: a
// context made after cudaDeviceReset gets a new one.
shkv_status current_context_id(unsigned long long *id)
{
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 12000);
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
    if (!get_current || !get_id)
        return SHKV_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS)
        return SHKV_ERR_CUDA;
    *id = 0;
    if (ctx && get_id(ctx, id) != CUDA_SUCCESS)
        return SHKV_ERR_CUDA;
    return SHKV_OK;
}

struct ScratchAddress {
    unsigned long long context_id;
    void *ptr;
};
std::mutex g_noalloc_mutex;
std::vector<ScratchAddress> g_noalloc_addresses;

// Device address of shkv_noalloc_scratch in the current context, looked up
// with cudaGetSymbolAddress the first time a context asks and cached by the
// context's unique ID.  (In host code the array's name is only a host-side
// stand-in, never a device address.)  A module loaded again in a new
// context -- after cudaDeviceReset, or in a context the caller made -- has
// its own scratch and its own entry.
shkv_status noalloc_scratch(void **ptr)
{
    unsigned long long id = 0;
    shkv_status st = current_context_id(&id);
    if (st != SHKV_OK)
        return st;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (id != 0)
        for (const ScratchAddress &a : g_noalloc_addresses)
            if (a.context_id == id) {
                *ptr = a.ptr;
                return SHKV_OK;
            }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, shkv_noalloc_scratch) != cudaSuccess || !p)
        return SHKV_ERR_CUDA;
    if (id == 0) {                       // the lookup made the primary context current
        st = current_context_id(&id);
        if (st != SHKV_OK || id == 0)
            return st != SHKV_OK ? st : SHKV_ERR_CUDA;
    }
    g_noalloc_addresses.push_back({id, p});
    *ptr = p;
    return SHKV_OK;
}

}  // namespace

extern "C" shkv_status shkv_decode_attention_noalloc(shkv_pool *pool, int32_t batch, int32_t n_models,
                                                     int32_t hq_per_model, const void *q, float scale, void *out,
                                                     float *lse_out, void *stream)
{
    if (!pool || !out)
        return SHKV_ERR_INVALID_ARG;
    if (batch < 1 || n_models < 1 || hq_per_model < 1)
        return SHKV_ERR_INVALID_ARG;
    if (hq_per_model % pool->cfg.num_kv_heads)
        return SHKV_ERR_UNSUPPORTED;
    // the scratch's counters are cleared by every call, so it takes only this
    // call's counters in front of the partials (the compact layout)
    const int32_t rows = n_models * (hq_per_model / pool->cfg.num_kv_heads);
    const size_t need = workspace_bytes_for(batch, pool->cfg.num_kv_heads, rows, pool->cfg.head_dim, pool->num_sms,
                                            /*compact=*/true);
    if (need > (size_t)SHKV_NOALLOC_SCRATCH_BYTES)
        return SHKV_ERR_UNSUPPORTED;
    shkv_status st;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess)
        return SHKV_ERR_CUDA;
    if (device != pool->device)
        return SHKV_ERR_INVALID_ARG;
    void *scratch = nullptr;
    st = noalloc_scratch(&scratch);
    if (st != SHKV_OK)
        return st;
    // decode_impl checks every argument first, then zeroes the arrival
    // counters at the front of the scratch on `stream`, then launches
    return decode_impl(pool, batch, n_models, hq_per_model, q, scale, out, lse_out, scratch, need, stream, nullptr,
                       /*clear_counters=*/true);
}
