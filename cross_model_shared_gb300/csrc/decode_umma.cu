// decode_umma.cu -- shared-KV decode attention on the 5th-generation tensor
// cores (tcgen05 / TMEM) for many stacked query rows per KV head (D = 128).
//
// Same method and work split as decode_attn.cu (ICaRus key design 3 over the
// PrefillShare paged cache: the N decoders' query rows of one KV head are
// stacked and share every K/V page load; persistent CTAs over cost-balanced
// chunk ranges; split units merged by the last arriving CTA).  Here tokens
// run along the MMA's M dimension.  A pipeline stage is 128 tokens of one
// (request, KV head), and per stage
//
//   S^T[t, r]  = sum_d K[t, d] Q[r, d]        M = 128 tokens,  N = rows
//   O^T[d, r] += sum_t V[t, d] P^T[t, r]      M = 128 = D,     N = rows
//
// so a TMEM lane is one token of S^T, or one head-dim column of O^T.  P is
// rounded to bf16 for the PV MMA; O is normalised by the sum of those same
// rounded weights (a row dominated by one token returns that token's V
// unchanged), and the log-sum-exp uses the fp32 sum of the unrounded ones.
// Roles (384 threads):
//
//   warps 0-7  softmax: warp w owns tokens 32*(w%4) .. +31 of each stage
//              (the TMEM lanes its sub-partition can reach) and half w/4 of
//              the stacked rows; each thread keeps fp32 row sums for its
//              token, reduced across the CTA at a segment end.  P^T (bf16)
//              is written over the stage's K tile, which the QK MMA no
//              longer needs; at 16 padded rows it has a buffer of its own
//              instead, so a slot's K half is refilled as soon as its QK
//              product completes.  At a segment end the same split reads O^T.
//   warp 8     QK issuer (one lane): S^T of each stage as soon as its data
//              has landed and an S buffer is free.
//   warp 9     K producer: TMA of each page's two K column halves (one copy
//              per lane) into a ring of 64 KiB stages, the query rows of the
//              next segment, and the validity word of each stage; for
//              32-token pages also the V halves.
//   warp 10    PV issuer (one lane): O^T of each stage as soon as its P is
//              written; its completion frees the ring slot.  (tcgen05.commit
//              tracks the issuing thread's MMAs, so the two issuers'
//              commits are independent.)
//   warp 11    V producer (16-token pages): TMA of each page's V halves.
//
// The running max m[r] is shared by all 128 tokens of a stage (O^T column r
// collects all of them), and it is refreshed lazily: every stage the eight
// warps vote, in one bar.red, whether any score exceeds m[r] + kRescaleLog2.
// Only then do they reduce the stage max across the CTA, rescale O^T in TMEM
// and the row sums in registers, and move m.  Unscaled exponentials stay
// below 2^kRescaleLog2.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "decode_common.cuh"
#include "launch.cuh"

namespace shkv {

namespace {

using namespace detail;

constexpr int kTT = 128;                    // tokens per stage (the MMA's M)
constexpr int kD = 128;                     // head dim (O^T's M)
constexpr int kHalves = kD / 64;            // 128-byte swizzle spans per row
constexpr int kTokenGroups = 4;             // 32-lane TMEM sub-partitions
constexpr int kSoftmaxWarps = 8;            // token group x row half
constexpr int kSoftmaxThreads = 32 * kSoftmaxWarps;
constexpr int kQkWarp = 8;
constexpr int kProducerWarp = 9;
constexpr int kPvWarp = 10;
constexpr int kVProducerWarp = 11;
constexpr int kTcThreads = 384;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;               // S^T buffers at columns 0 and 64
constexpr uint32_t kColO = 128;             // O^T
constexpr float kRescaleLog2 = 10.f;
constexpr int kTcMaxStages = 4;
// scratch rows of 64 floats: stage maxima [token group], new max, rescale
// factor, row-sum partials [token group] (rounded and exact), running max,
// the reciprocal rounded-weight row sum (one spare row keeps the layout)
constexpr int kScrMax = 0, kScrNew = 4, kScrAlpha = 5, kScrLhi = 6, kScrLex = 10, kScrM = 14, kScrSumHi = 15,
              kScrRows = 17;

static_assert(kTT == 32 * kTokenGroups, "one softmax thread per token of a stage and row half");
static_assert(kD == 32 * kTokenGroups, "one softmax thread per column of O^T and row half");

// Padded row count N of the MMAs for R stacked rows.
__host__ __device__ constexpr int tc_nr(int rows) { return (rows + 15) / 16 * 16; }
// N of the PV MMA: 48 is rounded up to a whole 64-column swizzle span.
__host__ __device__ constexpr int tc_npv(int nr) { return nr == 48 ? 64 : nr; }
// At 16 padded rows P^T has a buffer of its own (room for it beside a 3-slot
// ring exists only there), so a slot's K half is free once its QK product
// has completed and is refilled then, a PV product earlier than its V half.
__host__ __device__ constexpr bool tc_sep_p(int nr) { return nr == 16; }
// Entries of the validity-word ring when the K half is released early: the K
// producer runs at most 5 stages ahead of the softmax (3 K slots past the
// QK product, which is at most 2 S buffers past the softmax).
constexpr int kMetaRing = 8;
// Fused tails: the softmax needs each token's page word (valid tokens,
// attending decoder).  Up to 32 rows it loads the word from the unit's page
// word table itself, a stage ahead; above, where its registers are short,
// the K producer publishes a stage's words beside its validity word.
__host__ __device__ constexpr bool tc_words_by_producer(int nr) { return nr > 32; }

struct TcSmem {
    uint32_t ring, stage_bytes, qtile, qhalf, qbuf, qbuf_bytes, scr, rowoff, bars, meta, misc, tslot, total;
};

// Ring of `stages` slots of [K | V][half][128 tokens][128 B] (both 128-byte
// swizzled), with tc_sep_p the P^T buffer [128 tokens][128 B] (swizzled, as
// P^T over a K tile's first half), the Q tile [half][NR rows][128 B]
// (swizzled, K-major), one staging buffer of the next segment's query rows,
// the cross-warp scratch and the row-offset table, then the barriers and
// the validity words.
__host__ __device__ inline TcSmem tc_smem_layout(int rows, int stages, bool sep)
{
    TcSmem u;
    const int nr = tc_nr(rows);
    u.stage_bytes = (uint32_t)(2 * kTT * kD * 2);
    u.ring = 0;
    u.qhalf = (uint32_t)nr * 128u;
    u.qtile = u.ring + (uint32_t)stages * u.stage_bytes + (sep ? (uint32_t)(kTT * 128) : 0u);
    u.qbuf = u.qtile + (uint32_t)kHalves * u.qhalf;
    u.qbuf_bytes = align_up((uint32_t)(rows * kD * 2), 128);
    u.scr = u.qbuf + u.qbuf_bytes;
    u.rowoff = u.scr + (uint32_t)(kScrRows * 64 * 4);
    // full_k[stages], empty[stages], p_full[stages], full_v[stages], qfull,
    // qempty, s_full[2], s_free[2], q_ready, q_tile_free, fin; with tc_sep_p
    // also empty_k[stages], meta_full[kMetaRing]
    u.bars = align_up(u.rowoff + 64u * 4u, 8);
    u.meta = u.bars + (uint32_t)((4 * stages + 9 + (sep ? stages + kMetaRing : 0)) * 8);
    u.misc = u.meta + (uint32_t)((sep ? kMetaRing : stages) * kMetaWords * 4);
    u.tslot = u.misc + 8;
    u.total = u.misc + 16 + 1024;   // + slack to align the base to 1024 bytes
    return u;
}

struct TcCtx {
    uint8_t *smem;
    uint32_t base;
    TcSmem lay;
    int stages;
    volatile uint32_t *abort_flag;
    uint32_t *bcast;
    int64_t cta_begin, cta_end;
};

__device__ __forceinline__ uint32_t bar_at(const TcCtx &c, int i) { return c.base + c.lay.bars + 8u * i; }
// K (and the validity word) / V of the stage in ring slot s have landed.
__device__ __forceinline__ uint32_t full_b(const TcCtx &c, int s) { return bar_at(c, s); }
__device__ __forceinline__ uint32_t full_v_b(const TcCtx &c, int s) { return bar_at(c, 3 * c.stages + s); }
__device__ __forceinline__ uint32_t empty_b(const TcCtx &c, int s) { return bar_at(c, c.stages + s); }
// P of the stage in ring slot s is written (one phase per occupancy of the
// slot: the softmax reaches the slot's next stage only after PV freed it).
__device__ __forceinline__ uint32_t p_full_b(const TcCtx &c, int s) { return bar_at(c, 2 * c.stages + s); }
__device__ __forceinline__ uint32_t qfull_b(const TcCtx &c) { return bar_at(c, 4 * c.stages); }
__device__ __forceinline__ uint32_t qempty_b(const TcCtx &c) { return bar_at(c, 4 * c.stages + 1); }
__device__ __forceinline__ uint32_t s_full_b(const TcCtx &c, int b) { return bar_at(c, 4 * c.stages + 2 + b); }
__device__ __forceinline__ uint32_t s_free_b(const TcCtx &c, int b) { return bar_at(c, 4 * c.stages + 4 + b); }
__device__ __forceinline__ uint32_t q_ready_b(const TcCtx &c) { return bar_at(c, 4 * c.stages + 6); }
__device__ __forceinline__ uint32_t q_tile_free_b(const TcCtx &c) { return bar_at(c, 4 * c.stages + 7); }
__device__ __forceinline__ uint32_t fin_b(const TcCtx &c) { return bar_at(c, 4 * c.stages + 8); }
// (tc_sep_p) the K half of ring slot s is free: its QK product has completed
__device__ __forceinline__ uint32_t empty_k_b(const TcCtx &c, int s) { return bar_at(c, 4 * c.stages + 9 + s); }
// (tc_sep_p) validity-word entry i holds stage k (k % kMetaRing == i)
__device__ __forceinline__ uint32_t meta_b(const TcCtx &c, int i) { return bar_at(c, 5 * c.stages + 9 + i); }
__device__ __forceinline__ uint32_t slot_addr(const TcCtx &c, int slot)
{
    return c.base + c.lay.ring + (uint32_t)slot * c.lay.stage_bytes;
}
// Where P^T of a stage lives: over the stage's K tile (half 0), or (kSep)
// in the P buffer right after the ring.
template <bool kSep>
__device__ __forceinline__ uint32_t p_base(const TcCtx &c, uint32_t kst)
{
    if constexpr (kSep)
        return c.lay.ring + (uint32_t)c.stages * c.lay.stage_bytes;
    else
        return kst;
}
template <bool kSep>
__device__ __forceinline__ uint32_t p_tile(const TcCtx &c)
{
    return c.base + p_base<kSep>(c, c.lay.ring);
}
// descriptor offset (bytes >> 4) of K step ks of P^T: `off` for slot-resident P^T
template <bool kSep>
__device__ __forceinline__ uint32_t p_off(uint32_t off, int ks)
{
    if constexpr (kSep)
        return (uint32_t)ks * 128u;
    else
        return off;
}
// Entry of stage k's validity words: its slot, or (kSep) k % kMetaRing.
template <bool kSep>
__device__ __forceinline__ int meta_entry(int k, int slot)
{
    if constexpr (kSep)
        return k % kMetaRing;
    else
        return slot;
}

// A softmax thread's rows: 8-row chunks alternate between the two row
// halves, so element i of half hh is stacked row 16*(i/8) + 8*hh + i%8, and
// every TMEM access is 8 columns at a multiple of 8.
__device__ __forceinline__ int half_row(int hh, int i) { return ((i >> 3) << 4) + (hh << 3) + (i & 7); }

// This thread's N columns (N a multiple of 8) of a TMEM region starting at
// column `taddr`, as N/8 chunks of 8 at a stride of 16 from `taddr + 8*hh`.
template <int N>
__device__ __forceinline__ void tmem_ld_half(uint32_t taddr, int hh, uint32_t (&r)[N])
{
#pragma unroll
    for (int c = 0; c < N / 8; ++c)
        tmem_ld8_nowait(taddr + (uint32_t)(16 * c + 8 * hh), r + 8 * c);
    tmem_wait_ld();
}

template <int N>
__device__ __forceinline__ void tmem_st_half(uint32_t taddr, int hh, const uint32_t (&r)[N])
{
#pragma unroll
    for (int c = 0; c < N / 8; ++c)
        tmem_st8_nowait(taddr + (uint32_t)(16 * c + 8 * hh), r + 8 * c);
    tmem_wait_st();
}

// Warp reduce-scatter by recursive halving: at the butterfly step with lane
// offset O a lane keeps half of its M values and combines it with the
// partner's copy of that half.  Afterwards lane l holds in v[0 .. M/32 - 1]
// (v[0] if M < 32) the warp totals of columns rs_base<M>(l) + j; for M < 32,
// lanes that differ only in their low log2(32/M) bits hold the same column.
// M/2 + M/4 + ... shuffles instead of 5*M for a butterfly per column.
template <int M, int O, bool kMax>
struct ReduceScatter {
    static __device__ __forceinline__ void run(float *v, int lane)
    {
        if constexpr (O > 0) {
            if constexpr (M > 1) {
                const bool up = (lane & O) != 0;
#pragma unroll
                for (int i = 0; i < M / 2; ++i) {
                    const float send = up ? v[i] : v[i + M / 2];
                    const float keep = up ? v[i + M / 2] : v[i];
                    const float recv = __shfl_xor_sync(0xffffffffu, send, O);
                    v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
                }
                ReduceScatter<M / 2, O / 2, kMax>::run(v, lane);
            } else {
                const float recv = __shfl_xor_sync(0xffffffffu, v[0], O);
                v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
                ReduceScatter<1, O / 2, kMax>::run(v, lane);
            }
        }
    }
};

template <int M>
__device__ __forceinline__ int rs_base(int lane)
{
    int base = 0, m = M;
    for (int o = 16; o >= 1 && m > 1; o >>= 1) {
        if (lane & o)
            base += m / 2;
        m /= 2;
    }
    return base;
}

// lanes that hold a distinct column after a reduce-scatter of M values
template <int M>
__device__ __forceinline__ bool rs_owner(int lane)
{
    return M >= 32 || (lane & (32 / M - 1)) == 0;
}

__host__ __device__ constexpr int pow2_at_least(int n) { return n <= 8 ? 8 : n <= 16 ? 16 : n <= 32 ? 32 : 64; }

// ---------------------------------------------------------------------------
// producer warps
// ---------------------------------------------------------------------------
// Stage j of a segment is the 128 tokens from p0*P + j*128, i.e. 128/P
// pages.  Each page's two column halves of K and of V are copied with 2-D
// boxes of P rows x 128 B into [K | V][half][token][128 B] (the QK MMA reads
// 128 tokens of one half of K at a uniform stride, the PV MMA the same of V),
// one box per lane; K and V complete on separate full barriers, so QK starts
// as soon as K has landed.  With split_producers (16-token pages: 16 copies
// of each per stage) the K warp copies K, the query rows and the validity
// word while the V warp copies V; otherwise (8 of each) the K warp issues
// all of them, K first, and the V warp has nothing to do (measured faster).
template <bool kIsK, bool kSep, bool kWords>
__device__ void tc_producer(const CUtensorMap *tmK, const CUtensorMap *tmV, const DecodeParams &p, const TcCtx &c)
{
    const int lane = threadIdx.x & 31;
    const int stages = c.stages;
    const int P = p.page_size;
    const int RB = kTT / P;                              // pages per stage (4 or 8)
    const int log2P = 31 - __clz(P);
    const bool split = p.split_producers != 0;
    if (!kIsK && !split)
        return;
    // lane -> (tensor, half, page): K lanes first, then V lanes when one warp copies both
    const int per_tensor = kHalves * RB;
    const bool my_v = kIsK ? lane >= per_tensor : true;
    const int cl = (my_v && kIsK) ? lane - per_tensor : lane;
    const int my_h = cl / RB;
    const int my_rb = cl % RB;
    const bool copier = kIsK ? (lane < (split ? per_tensor : 2 * per_tensor)) : lane < per_tensor;
    const uint32_t page_bytes = kHalves * (uint32_t)P * 128u;   // K or V of one page
    const uint64_t pol = l2_evict_first_policy();
    if (lane == 0) {
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
    }

    bool alive = true;
    int kbase = 0, seg = 0;
    int last_issued_stage = -1;
    int q_issued = -1;
    Segment s = locate(p, c.cta_begin, c.cta_end);
    int pre = unit_entry(p.block_table, p, s.b, s.p0 + lane, s.p1);
    // kWords (fused tails, the K warp): page words, in windows like the ids
    constexpr bool words = kWords && kIsK;
    const int32_t *info_tab = reinterpret_cast<const int32_t *>(p.page_info);
    int pre_i = words ? unit_entry(info_tab, p, s.b, s.p0 + lane, s.p1) : -1;
    for (;;) {
        const bool has_next = s.seg_end < c.cta_end;
        Segment sn;
        int pre_next = -1, pre_next_i = -1;
        if (has_next) {
            sn = next_segment(p, s, c.cta_end);
            pre_next = unit_entry(p.block_table, p, sn.b, lane, sn.p1);
            if constexpr (words)
                pre_next_i = unit_entry(info_tab, p, sn.b, lane, sn.p1);
        }
        // (a unit of fused tails is not one sequence: no length to check)
        const int dev_len = (kIsK && lane == 0 && p.fused == 0) ? __ldg(p.seq_lens + s.b) : 0;
        // --- query rows of this (b, g): N bulk copies of G contiguous rows
        if (kIsK) {
            if (alive) {
                bool ok = mbar_wait_bounded(qempty_b(c), (uint32_t)((seg & 1) ^ 1), c.abort_flag, p.err);
                alive = __all_sync(0xffffffffu, ok);
            }
            if (alive && lane == 0) {
                const uint32_t rows_bytes = (uint32_t)p.group * kD * 2u;
                mbar_arrive_expect_tx(qfull_b(c), rows_bytes * p.n_models);
                const __nv_bfloat16 *qsrc =
                    p.q + ((int64_t)s.b * p.n_models * p.hq + (int64_t)s.g * p.group) * kD;
                const uint32_t qdst = c.base + c.lay.qbuf;
                for (int m = 0; m < p.n_models; ++m)
                    bulk_load(qdst + m * rows_bytes, qsrc + (int64_t)m * p.hq * kD, rows_bytes, qfull_b(c));
                q_issued = seg;
            }
        }
        // --- K or V pages of the segment
        const int tok_end = s.p1 * P;
        const int nst = (tok_end - s.p0 * P + kTT - 1) / kTT;
        const int32_t *btrow = p.block_table + (int64_t)s.b * p.max_pages;
        int w0 = s.p0;                                   // block-table window [w0, w0+32)
        int cur = pre, cur_i = pre_i;
        int nxt = (w0 + 32 + lane < s.p1) ? __ldg(btrow + w0 + 32 + lane) : -1;
        int nxt_i = words ? unit_entry(info_tab, p, s.b, w0 + 32 + lane, s.p1) : -1;
        for (int j = 0; j < nst; ++j) {
            const int k = kbase + j;
            const int slot = k % stages;
            const int tok0 = s.p0 * P + j * kTT;
            // a stage's pages start at a multiple of RB from p0, so they never
            // straddle a 32-entry window
            if ((tok0 >> log2P) >= w0 + 32) {
                w0 += 32;
                cur = nxt;
                nxt = (w0 + 32 + lane < s.p1) ? __ldg(btrow + w0 + 32 + lane) : -1;
                if constexpr (words) {
                    cur_i = nxt_i;
                    nxt_i = unit_entry(info_tab, p, s.b, w0 + 32 + lane, s.p1);
                }
            }
            const int my_tok = tok0 + my_rb * P;
            const int my_id = __shfl_sync(0xffffffffu, cur, ((my_tok >> log2P) - w0) & 31);
            // (words) page word of page rb of the stage, gathered to lane 0 (lane rb < RB holds page rb)
            uint32_t pinfo[8];
            if constexpr (words) {
                const int my_info = __shfl_sync(0xffffffffu, cur_i, ((my_tok >> log2P) - w0) & 31);
#pragma unroll
                for (int rb = 0; rb < 8; ++rb)
                    pinfo[rb] = (uint32_t)__shfl_sync(0xffffffffu, my_info, rb);
            }
            bool ok = true;
            if constexpr (kSep && kIsK) {
                // the K warp of split producers refills a slot's K half once QK freed it
                if (alive)
                    ok = mbar_wait_bounded(split ? empty_k_b(c, slot) : empty_b(c, slot),
                                           (uint32_t)(((k / stages) & 1) ^ 1), c.abort_flag, p.err);
            } else {
                if (alive)  // every lane polls (measured faster than one lane and a warp barrier)
                    ok = mbar_wait_bounded(empty_b(c, slot), (uint32_t)(((k / stages) & 1) ^ 1), c.abort_flag, p.err);
            }
            alive = alive && __all_sync(0xffffffffu, ok);
            const bool my_valid = copier && my_tok < tok_end && my_id >= 0 && my_id < p.num_pages;
            // lanes 0..RB-1 copy page rb = lane (half 0 for K): their ballot is the page mask
            const uint32_t mask = __ballot_sync(0xffffffffu, my_valid) & ((1u << RB) - 1u);
            if (alive && lane == 0) {
                if (kIsK) {
                    for (int rb = 0; rb < RB; ++rb)
                        if (!((mask >> rb) & 1u) && tok0 + rb * P < tok_end)
                            atomicOr(p.err, SHKV_ERRF_PAGE_OOB);
                    volatile uint32_t *meta =
                        reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.meta) + meta_entry<kSep>(k, slot) * kMetaWords;
                    if constexpr (words) {
#pragma unroll
                        for (int rb = 0; rb < 8; ++rb)
                            if (rb < RB)
                                meta[1 + rb] = pinfo[rb];
                    }
                    meta[0] = mask | ((uint32_t)k << 8);   // valid pages + stage tag
                    if constexpr (kSep)
                        mbar_arrive(meta_b(c, k % kMetaRing));
                    mbar_arrive_expect_tx(full_b(c, slot), (uint32_t)__popc(mask) * page_bytes);
                }
                if (!kIsK || !split)
                    mbar_arrive_expect_tx(full_v_b(c, slot), (uint32_t)__popc(mask) * page_bytes);
            }
            __syncwarp();
            if (alive && my_valid) {
                const uint32_t dst = slot_addr(c, slot) + (my_v ? (uint32_t)(kTT * kD * 2) : 0u) +
                                     (uint32_t)my_h * (kTT * 128) + (uint32_t)my_rb * (uint32_t)P * 128u;
                tma_load_2d(dst, my_v ? tmV : tmK, my_h * 64, (my_id * p.hkv + s.g) * P,
                            my_v ? full_v_b(c, slot) : full_b(c, slot), pol);
            }
            if (alive)
                last_issued_stage = k;
            __syncwarp();
        }
        if (kIsK && lane == 0 && p.fused == 0 && dev_len != plan_len(p, s))
            atomicOr(p.err, SHKV_ERRF_SEQ_LEN);
        kbase += nst;
        ++seg;
        if (!has_next)
            break;
        s = sn;
        pre = pre_next;
        pre_i = pre_next_i;
    }
    // After an abort, wait (bounded) for the copies still in flight so no TMA
    // write lands after the CTA exits.
    if (!alive && lane == 0) {
        for (int k = last_issued_stage - stages + 1; k <= last_issued_stage; ++k)
            if (k >= 0) {
                if (kIsK)
                    mbar_drain_bounded(full_b(c, k % stages), (uint32_t)((k / stages) & 1));
                if (!kIsK || !split)
                    mbar_drain_bounded(full_v_b(c, k % stages), (uint32_t)((k / stages) & 1));
            }
        if (q_issued >= 0)
            mbar_drain_bounded(qfull_b(c), (uint32_t)(q_issued & 1));
    }
}

// Run by the producer warps before they wait for the previous grid: prefetch
// into L2 the page halves of this CTA's first ring-full of stages (up to 32
// pages of its first segment; K from the K warp, V from the warp that will
// copy it), so that the first copies after the wait hit L2 instead of waiting
// on DRAM.  The block-table entries are read through L2 only and may be
// stale (a preceding kernel may still be writing them): they are used for
// nothing but these prefetches, and an id outside the pool is skipped.
template <bool kIsK>
__device__ void tc_warm_l2(const CUtensorMap *tmK, const CUtensorMap *tmV, const DecodeParams &p, const TcCtx &c)
{
    const int lane = threadIdx.x & 31;
    const bool split = p.split_producers != 0;
    if (!kIsK && !split)
        return;
    const Segment s = locate(p, c.cta_begin, c.cta_end);
    const int P = p.page_size;
    const int ring_pages = c.stages * kTT / P;
    const int pages = s.p1 - s.p0 < ring_pages ? s.p1 - s.p0 : ring_pages;
    if (lane < pages) {
        const int id = __ldcg(p.block_table + (int64_t)s.b * p.max_pages + s.p0 + lane);
        if (id >= 0 && id < p.num_pages) {
            const int y = (id * p.hkv + s.g) * P;
#pragma unroll
            for (int h = 0; h < kHalves; ++h) {
                if (kIsK)
                    tma_prefetch_2d(tmK, h * 64, y);
                if (!kIsK || !split)
                    tma_prefetch_2d(tmV, h * 64, y);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// MMA issuers (one lane each)
// ---------------------------------------------------------------------------
// The descriptors of a stage are built before its waits end, so that once
// the data is there the issue is only the MMA instructions (the issuing
// thread shares its SM sub-partition with two softmax warps).  Each operand
// has one base descriptor; the others add (byte offset >> 4) to its 14-bit
// address field, which shared addresses below 256 KB never carry out of.
template <int NR>
__device__ void tc_qk(const DecodeParams &p, const TcCtx &c, uint32_t tmem)
{
    constexpr bool kSep = tc_sep_p(NR);
    const int stages = c.stages;
    const int P = p.page_size;
    const uint32_t idesc_qk = umma_idesc_bf16(128, NR, false, false);
    uint64_t bq[kHalves * 4];                 // the Q tile (B), K-major
#pragma unroll
    for (int i = 0; i < kHalves * 4; ++i)
        bq[i] = umma_sdesc_sw128(c.base + c.lay.qtile + (uint32_t)(i >> 2) * c.lay.qhalf + (uint32_t)((i & 3) * 32),
                                 16u, 1024u);
    const uint64_t kd0 = umma_sdesc_sw128(slot_addr(c, 0), 16u, 1024u);
    bool alive = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (alive)
            alive = mbar_wait_bounded(bar, parity, c.abort_flag, p.err);
        return alive;
    };
    int kbase = 0, seg = 0;
    Segment s = locate(p, c.cta_begin, c.cta_end);
    for (;;) {
        const int nst = (s.p1 * P - s.p0 * P + kTT - 1) / kTT;
        wait(q_ready_b(c), (uint32_t)(seg & 1));
        tc_fence_after();
        for (int j = 0; j < nst; ++j) {
            const int k = kbase + j;
            const int buf = k & 1;
            const int slot = k % stages;
            uint64_t ak[kHalves * 4];         // this stage's K tile (A), K-major
#pragma unroll
            for (int i = 0; i < kHalves * 4; ++i)
                ak[i] = kd0 + (((uint32_t)slot * c.lay.stage_bytes + (uint32_t)((i >> 2) * kTT * 128 + (i & 3) * 32)) >> 4);
            wait(full_b(c, slot), (uint32_t)((k / stages) & 1));
            wait(s_free_b(c, buf), (uint32_t)(((k >> 1) & 1) ^ 1));
            if (alive) {
                tc_fence_after();
                const uint32_t d = tmem + kColS + (uint32_t)(buf * 64);
#pragma unroll
                for (int i = 0; i < kHalves * 4; ++i)
                    umma_bf16(d, ak[i], bq[i], idesc_qk, i ? 1u : 0u);
            }
            umma_commit(s_full_b(c, buf));
            if constexpr (kSep)
                umma_commit(empty_k_b(c, slot));
            if (j == nst - 1)
                umma_commit(q_tile_free_b(c));
        }
        kbase += nst;
        ++seg;
        if (s.seg_end >= c.cta_end)
            break;
        s = next_segment(p, s, c.cta_end);
    }
    // every MMA this thread issued has completed once fin's phase ends
    umma_commit(fin_b(c));
    mbar_drain_bounded(fin_b(c), 0u);
}

// O^T += V^T P^T for each stage; P^T sits over the stage's K tile (half 0),
// or in the P buffer (sep_p).
template <int NR>
__device__ void tc_pv(const DecodeParams &p, const TcCtx &c, uint32_t tmem)
{
    constexpr bool kSep = tc_sep_p(NR);
    constexpr int NPV = tc_npv(NR);
    const int stages = c.stages;
    const int P = p.page_size;
    const uint32_t idesc_pv = umma_idesc_bf16(128, NPV, true, true);
    // V^T (A) and P^T (B, over the K tile's first half or in the P buffer), both MN-major
    const uint64_t vd0 = umma_sdesc_sw128(slot_addr(c, 0) + (uint32_t)(kTT * kD * 2), (uint32_t)(kTT * 128), 1024u);
    const uint64_t pd0 = umma_sdesc_sw128(p_tile<kSep>(c), (uint32_t)(kTT * 128), 1024u);
    bool alive = true;
    int kbase = 0;
    Segment s = locate(p, c.cta_begin, c.cta_end);
    for (;;) {
        const int nst = (s.p1 * P - s.p0 * P + kTT - 1) / kTT;
        for (int j = 0; j < nst; ++j) {
            const int k = kbase + j;
            const int slot = k % stages;
            uint64_t av[kTT / 16], bp[kTT / 16];
#pragma unroll
            for (int ks = 0; ks < kTT / 16; ++ks) {
                const uint32_t off = ((uint32_t)slot * c.lay.stage_bytes + (uint32_t)ks * 2048u) >> 4;
                av[ks] = vd0 + off;
                bp[ks] = pd0 + p_off<kSep>(off, ks);
            }
            if (alive)
                alive = mbar_wait_bounded(p_full_b(c, slot), (uint32_t)((k / stages) & 1), c.abort_flag, p.err);
            if (alive)
                alive = mbar_wait_bounded(full_v_b(c, slot), (uint32_t)((k / stages) & 1), c.abort_flag, p.err);
            if (alive) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < kTT / 16; ++ks)
                    umma_bf16(tmem + kColO, av[ks], bp[ks], idesc_pv, (j == 0 && ks == 0) ? 0u : 1u);
            }
            umma_commit(empty_b(c, slot));
        }
        kbase += nst;
        if (s.seg_end >= c.cta_end)
            break;
        s = next_segment(p, s, c.cta_end);
    }
    umma_commit(fin_b(c));
    mbar_drain_bounded(fin_b(c), 0u);
}

// ---------------------------------------------------------------------------
// softmax warps
// ---------------------------------------------------------------------------
// Thread (warp w, lane l): token / O^T column t = 32*(w%4) + l, and the
// stacked rows half_row(w/4, i) for i < NR/2.
template <int NR, bool FUSED>
__device__ void tc_softmax(const DecodeParams &p, const TcCtx &c, uint32_t tmem)
{
    constexpr bool kSep = tc_sep_p(NR);
    constexpr int NH = NR / 2;                 // rows per thread
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tg = warp & (kTokenGroups - 1);
    const int hh = warp / kTokenGroups;
    const int t = tg * 32 + lane;
    const int stages = c.stages;
    const int P = p.page_size;
    const int R = p.rows;
    const int log2P = 31 - __clz(P);
    const float sl2 = p.scale_log2;
    const uint32_t lane_base = (uint32_t)(tg * 32) << 16;
    const volatile uint32_t *meta = reinterpret_cast<const volatile uint32_t *>(c.smem + c.lay.meta);
    float *scr = reinterpret_cast<float *>(c.smem + c.lay.scr);
    const int *rowoff = reinterpret_cast<const int *>(c.smem + c.lay.rowoff);
    bool alive = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        bool ok = false;
        if (alive)
            ok = mbar_wait_bounded(bar, parity, c.abort_flag, p.err);
        alive = __all_sync(0xffffffffu, ok) && alive;
        return alive;
    };

    // query rows of segment `sg`: staging buffer -> swizzled K-major Q tile
    auto stage_q = [&](int sg) {
        wait(qfull_b(c), (uint32_t)(sg & 1));
        if (alive) {
            const uint8_t *src = c.smem + c.lay.qbuf;
            for (int e = threadIdx.x; e < R * (kD / 8); e += kSoftmaxThreads) {
                const int rr = e >> 4, ch = e & 15;
                const uint4 v = *reinterpret_cast<const uint4 *>(src + rr * (kD * 2) + ch * 16);
                const uint32_t off = (uint32_t)(ch >> 3) * c.lay.qhalf + (uint32_t)rr * 128u +
                                     (uint32_t)(((ch & 7) ^ (rr & 7)) << 4);
                *reinterpret_cast<uint4 *>(c.smem + c.lay.qtile + off) = v;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(qempty_b(c));
            mbar_arrive(q_ready_b(c));
        }
    };

    int kbase = 0, seg = 0;
    Segment s = locate(p, c.cta_begin, c.cta_end);
    stage_q(0);
    for (;;) {
        const int tok_end = s.p1 * P;
        const int nst = (tok_end - s.p0 * P + kTT - 1) / kTT;
        constexpr bool fused = FUSED;
        const int L = fused ? tok_end : plan_len(p, s);   // fused tails: valid tokens per page from page_info
        const int lim = L < tok_end ? L : tok_end;
        // fused tails: this thread's token's page word (valid tokens, decoder)
        // for stage jj, read through L2 (the unit kernel wrote it) a stage
        // ahead of its use
        auto page_word = [&](int jj) -> uint32_t {
            const int pg = s.p0 + ((jj * kTT + t) >> log2P);
            return jj < nst && pg < s.p1
                       ? __ldcg(reinterpret_cast<const uint32_t *>(p.page_info) + (int64_t)s.b * p.max_pages + pg)
                       : 0u;
        };
        constexpr bool own_words = fused && !tc_words_by_producer(NR);
        uint32_t tinfo_next = own_words ? page_word(0) : (kAllDecoders << 8);
        float m_use[NH], lhi[NH], lex[NH];
#pragma unroll
        for (int i = 0; i < NH; ++i) {
            m_use[i] = -INFINITY;
            lhi[i] = 0.f;
            lex[i] = 0.f;
        }

        for (int j = 0; j < nst; ++j) {
            const int k = kbase + j;
            const int buf = k & 1;
            const int slot = k % stages;
            // --- this token's scores for this thread's rows
            uint32_t sv[NH];
            if (wait(s_full_b(c, buf), (uint32_t)((k >> 1) & 1))) {
                tc_fence_after();
                tmem_ld_half<NH>(tmem + lane_base + kColS + (uint32_t)(buf * 64), hh, sv);
            } else {
#pragma unroll
                for (int i = 0; i < NH; ++i)
                    sv[i] = 0u;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(s_free_b(c, buf));
            // the stage's validity word (the QK MMA has already consumed the data);
            // with sep_p the slot's K barrier may already be a phase further on
            const int mi = meta_entry<kSep>(k, slot);
            if constexpr (kSep)
                wait(meta_b(c, mi), (uint32_t)((k / kMetaRing) & 1));
            else
                wait(full_b(c, slot), (uint32_t)((k / stages) & 1));
            const uint32_t tagged = alive ? meta[mi * kMetaWords] : 0u;
            if (alive && (tagged >> 8) != ((uint32_t)k & 0xffffffu)) {
                if (lane == 0) {
                    atomicOr(p.err, SHKV_ERRF_PIPELINE);
                    *c.abort_flag = 1u;
                }
                alive = false;
            }
            const int tok0 = s.p0 * P + j * kTT;
            uint32_t tinfo = tinfo_next;
            if constexpr (own_words)
                tinfo_next = page_word(j + 1);
            else if constexpr (fused)
                tinfo = alive ? meta[mi * kMetaWords + 1 + (t >> log2P)] : (kAllDecoders << 8);
            const uint32_t tdec = (tinfo >> 8) & 0xffu;
            const bool valid = alive && (((tagged & 0xffu) >> (t >> log2P)) & 1u) &&
                               (fused ? (uint32_t)(t & (P - 1)) < (tinfo & 0xffu) : (tok0 + t < lim));
            const uint32_t kst = c.lay.ring + (uint32_t)slot * c.lay.stage_bytes;
            // rows past the length inside a copied page are written by the V
            // copy: zero them only after it has landed
            if (__any_sync(0xffffffffu, alive && !valid))
                wait(full_v_b(c, slot), (uint32_t)((k / stages) & 1));
            if (alive && !valid) {
                // this token's V row (this warp's column half) may hold stale
                // or non-finite bits: zero it
                const uint32_t vrow =
                    c.base + kst + (uint32_t)(kTT * kD * 2) + (uint32_t)(hh * kTT * 128) + (uint32_t)t * 128u;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    st_shared_zero16(vrow + (uint32_t)(ch * 16));
            }
            float xs[NH];
            bool need = false;
#pragma unroll
            for (int i = 0; i < NH; ++i) {
                // a tail page is attended by its decoder's rows only
                const bool attends =
                    tdec == kAllDecoders || (uint32_t)(half_row(hh, i) - (int)tdec * p.group) < (uint32_t)p.group;
                xs[i] = valid && attends ? __uint_as_float(sv[i]) * sl2 : -INFINITY;
                need = need || (xs[i] > m_use[i] + kRescaleLog2);
            }
            // --- lazy max refresh: the eight warps agree on a new m[] together
            if (bar_red_or(1, kSoftmaxThreads, need)) {
                {
                    constexpr int M = pow2_at_least(NH);
                    float v[M];
#pragma unroll
                    for (int i = 0; i < M; ++i)
                        v[i] = i < NH ? xs[i] : -INFINITY;
                    ReduceScatter<M, 16, true>::run(v, lane);
                    const int base = rs_base<M>(lane);
                    if (rs_owner<M>(lane))
#pragma unroll
                        for (int j = 0; j < (M >= 32 ? M / 32 : 1); ++j)
                            if (base + j < NH)
                                scr[(kScrMax + tg) * 64 + half_row(hh, base + j)] = v[j];
                }
                named_barrier(1, kSoftmaxThreads);
                if (threadIdx.x < NR) {
                    const int r = threadIdx.x;
                    const float mo = scr[kScrM * 64 + r];
                    float mn = mo;
#pragma unroll
                    for (int g = 0; g < kTokenGroups; ++g)
                        mn = fmaxf(mn, scr[(kScrMax + g) * 64 + r]);
                    scr[kScrNew * 64 + r] = mn;
                    scr[kScrAlpha * 64 + r] = mn == -INFINITY ? 1.f : ex2_approx(mo - mn);
                    scr[kScrM * 64 + r] = mn;
                }
                named_barrier(1, kSoftmaxThreads);
                const float *alpha = scr + kScrAlpha * 64;
                if (j >= 1) {
                    // O^T holds stages up to k-1: rescale this thread's part once PV(k-1) is done
                    const int kp = k - 1;
                    wait(empty_b(c, kp % stages), (uint32_t)((kp / stages) & 1));
                    if (alive) {
                        tc_fence_after();
                        uint32_t ov[NH];
                        tmem_ld_half<NH>(tmem + lane_base + kColO, hh, ov);
#pragma unroll
                        for (int i = 0; i < NH; ++i)
                            ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha[half_row(hh, i)]);
                        tmem_st_half<NH>(tmem + lane_base + kColO, hh, ov);
                    }
                }
#pragma unroll
                for (int i = 0; i < NH; ++i) {
                    m_use[i] = scr[kScrNew * 64 + half_row(hh, i)];
                    lhi[i] *= alpha[half_row(hh, i)];
                    lex[i] *= alpha[half_row(hh, i)];
                }
            }
            // --- this token's part of P^T, over the stage's K tile (half 0) or, with
            // sep_p, in the P buffer once the previous stage's PV has read it
            if constexpr (kSep) {
                if (k > 0)
                    wait(empty_b(c, (k - 1) % stages), (uint32_t)(((k - 1) / stages) & 1));
            }
            uint8_t *prow = c.smem + p_base<kSep>(c, kst) + (uint32_t)t * 128u;
#pragma unroll
            for (int ch = 0; ch < NH / 8; ++ch) {
                uint32_t hi[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = ch * 8 + 2 * e;
                    const float mu0 = m_use[i] == -INFINITY ? 0.f : m_use[i];
                    const float mu1 = m_use[i + 1] == -INFINITY ? 0.f : m_use[i + 1];
                    const float p0 = ex2_approx(xs[i] - mu0);
                    const float p1 = ex2_approx(xs[i + 1] - mu1);
                    hi[e] = pack_bf16x2(p0, p1);
                    lex[i] += p0;
                    lex[i + 1] += p1;
                    lhi[i] += __uint_as_float(hi[e] << 16);
                    lhi[i + 1] += __uint_as_float(hi[e] & 0xffff0000u);
                }
                if (alive) {
                    const int gch = 2 * ch + hh;
                    *reinterpret_cast<uint4 *>(prow + ((gch ^ (t & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(p_full_b(c, slot));
        }

        // --- next segment's query rows, as soon as the last QK of this one is done
        const bool has_next = s.seg_end < c.cta_end;
        if (has_next) {
            wait(q_tile_free_b(c), (uint32_t)(seg & 1));
            stage_q(seg + 1);
        }

        // --- segment end: row sums across the 128 tokens, log-sum-exp
        {
            constexpr int M = pow2_at_least(2 * NH);
            float v[M];
#pragma unroll
            for (int i = 0; i < M; ++i)
                v[i] = i < NH ? lhi[i] : i < 2 * NH ? lex[i - NH] : 0.f;
            ReduceScatter<M, 16, false>::run(v, lane);
            const int base = rs_base<M>(lane);
            if (rs_owner<M>(lane))
#pragma unroll
                for (int j = 0; j < (M >= 32 ? M / 32 : 1); ++j) {
                    const int col = base + j;
                    if (col < NH)
                        scr[(kScrLhi + tg) * 64 + half_row(hh, col)] = v[j];
                    else if (col < 2 * NH)
                        scr[(kScrLex + tg) * 64 + half_row(hh, col - NH)] = v[j];
                }
        }
        named_barrier(1, kSoftmaxThreads);
        const bool whole = (s.seg_begin == s.unit_begin) && (s.seg_end == s.unit_end);
        const int slot_id = whole ? 0 : 2 * (int)blockIdx.x + (s.seg_begin == c.cta_begin ? 0 : 1);
        const int64_t row0 = (int64_t)s.b * p.n_models * p.hq + (int64_t)s.g * p.group;
        if (threadIdx.x < NR) {
            const int r = threadIdx.x;
            float a = 0.f, b = 0.f;
#pragma unroll
            for (int g = 0; g < kTokenGroups; ++g) {
                a += scr[(kScrLhi + g) * 64 + r];
                b += scr[(kScrLex + g) * 64 + r];
            }
            scr[kScrSumHi * 64 + r] = a > 0.f ? __frcp_rn(a) : 0.f;   // 1 / row sum, for O
            const float m = scr[kScrM * 64 + r];
            scr[kScrM * 64 + r] = -INFINITY;        // the next segment starts afresh
            if (alive && r < R) {
                const float lse = b > 0.f ? (m + log2f(b)) * kLn2 : -INFINITY;
                if (whole) {
                    if (p.lse_out)
                        p.lse_out[row0 + rowoff[r]] = lse;
                } else {
                    p.ws_lse[(int64_t)slot_id * R + r] = lse;
                }
            }
        }
        named_barrier(1, kSoftmaxThreads);

        // --- column d = t of O^T for this thread's rows, normalised
        const int last = kbase + nst - 1;
        wait(empty_b(c, last % stages), (uint32_t)((last / stages) & 1));
        if (alive) {
            tc_fence_after();
            uint32_t ov[NH];
            tmem_ld_half<NH>(tmem + lane_base + kColO, hh, ov);
#pragma unroll
            for (int i = 0; i < NH; ++i) {
                const int r = half_row(hh, i);
                if (r < R) {
                    const float o = __uint_as_float(ov[i]) * scr[kScrSumHi * 64 + r];
                    if (!whole)
                        p.ws_part[((int64_t)slot_id * R + r) * kD + t] = o;
                    else
                        p.out[(row0 + rowoff[r]) * kD + t] = __float2bfloat16_rn(o);
                }
            }
        }
        tc_fence_before();
        named_barrier(1, kSoftmaxThreads);

        // --- split unit: the last piece to arrive merges all pieces
        if (!whole) {
            const int cb = cta_of(p, s.unit_begin);
            const int ce = cta_of(p, s.unit_end - 1);
            uint32_t *counter = p.ws_count + (int64_t)s.b * p.hkv + s.g;
            if (threadIdx.x == 0) {
                __threadfence();
                const uint32_t prev = atomicAdd(counter, 1u);
                *c.bcast = (prev == (uint32_t)(ce - cb)) ? 1u : 0u;
            }
            named_barrier(1, kSoftmaxThreads);
            if (*c.bcast) {
                __threadfence();
                const int dq = kD / 4;
                for (int rr = warp; rr < R; rr += kSoftmaxWarps) {
                    float M = -INFINITY;
                    for (int cc = cb + lane; cc <= ce; cc += 32)
                        M = fmaxf(M, __ldcg(p.ws_lse + (int64_t)piece_slot(p, cc, s.unit_begin) * R + rr));
#pragma unroll
                    for (int o_ = 16; o_ > 0; o_ >>= 1)
                        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o_));
                    float wsum = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (M != -INFINITY) {
                        for (int cc = cb; cc <= ce; ++cc) {
                            const int sl = piece_slot(p, cc, s.unit_begin);
                            const float w = ex2_approx((__ldcg(p.ws_lse + (int64_t)sl * R + rr) - M) *
                                                       1.4426950408889634f);
                            wsum += w;
                            if (lane < dq) {
                                const float4 v = __ldcg(
                                    reinterpret_cast<const float4 *>(p.ws_part + ((int64_t)sl * R + rr) * kD) + lane);
                                acc.x += w * v.x;
                                acc.y += w * v.y;
                                acc.z += w * v.z;
                                acc.w += w * v.w;
                            }
                        }
                    }
                    const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
                    const int64_t orr = row0 + rowoff[rr];
                    if (lane < dq) {
                        uint2 packed;
                        packed.x = pack_bf16x2(acc.x * winv, acc.y * winv);
                        packed.y = pack_bf16x2(acc.z * winv, acc.w * winv);
                        *reinterpret_cast<uint2 *>(p.out + orr * kD + lane * 4) = packed;
                    }
                    if (lane == 0 && p.lse_out)
                        p.lse_out[orr] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
                }
                if (threadIdx.x == 0)
                    *counter = 0u;
            }
            named_barrier(1, kSoftmaxThreads);
        }

        kbase += nst;
        ++seg;
        if (!has_next)
            break;
        s = next_segment(p, s, c.cta_end);
    }
}

}  // namespace

// 12 warps at one CTA per SM: three warps share a 16K-register SM
// sub-partition, so at most 168 registers a thread.
template <int NR, bool FUSED>
__global__ void __launch_bounds__(kTcThreads, 1)
    shkv_decode_umma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    TcCtx c;
    {
        const uint32_t raw = smem_u32(smem_raw);
        const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
        c.smem = smem_raw + pad;
        c.base = raw + pad;
    }
    c.stages = p.stages;
    c.lay = tc_smem_layout(p.rows, p.stages, tc_sep_p(NR));
    c.abort_flag = reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.misc);
    c.bcast = reinterpret_cast<uint32_t *>(c.smem + c.lay.misc + 4);
    c.cta_begin = p.cta_cut[blockIdx.x];
    c.cta_end = p.cta_cut[blockIdx.x + 1];
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < c.stages; ++s) {
            mbar_init(full_b(c, s), 1);
            mbar_init(full_v_b(c, s), 1);
            mbar_init(empty_b(c, s), 1);                     // one tcgen05.commit per stage
            mbar_init(p_full_b(c, s), kSoftmaxWarps);
        }
        mbar_init(qfull_b(c), 1);
        mbar_init(qempty_b(c), kSoftmaxWarps);
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full_b(c, i), 1);
            mbar_init(s_free_b(c, i), kSoftmaxWarps);
        }
        mbar_init(q_ready_b(c), kSoftmaxWarps);
        mbar_init(q_tile_free_b(c), 1);
        mbar_init(fin_b(c), 2);                              // one commit per MMA issuer
        if constexpr (tc_sep_p(NR)) {
            for (int s = 0; s < c.stages; ++s)
                mbar_init(empty_k_b(c, s), 1);               // the QK product's commit
            for (int i = 0; i < kMetaRing; ++i)
                mbar_init(meta_b(c, i), 1);                  // the K producer
        }
        *c.abort_flag = 0u;
        *c.bcast = 0u;
        fence_barrier_init();
    }
    if (warp < kSoftmaxWarps) {
        // zeroed Q tile (its padding rows stay zero), running maxima, row offsets
        for (uint32_t i = threadIdx.x; i < (uint32_t)kHalves * c.lay.qhalf / 16; i += kSoftmaxThreads)
            *reinterpret_cast<uint4 *>(c.smem + c.lay.qtile + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
        if (threadIdx.x < 64) {
            const int r = threadIdx.x;
            reinterpret_cast<float *>(c.smem + c.lay.scr)[kScrM * 64 + r] = -INFINITY;
            const int m = r / p.group, jj = r - (r / p.group) * p.group;
            reinterpret_cast<int *>(c.smem + c.lay.rowoff)[r] = m * p.hq + jj;
        }
        fence_proxy_async_smem();
    }
    if (warp == 0)
        tmem_alloc(c.base + c.lay.tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.tslot);
    if (warp == kProducerWarp)
        tc_warm_l2<true>(&tmK, &tmV, p, c);
    else if (warp == kVProducerWarp)
        tc_warm_l2<false>(&tmK, &tmV, p, c);
    pdl_wait_prior();                       // global memory only from here on
    pdl_launch_dependents();                // (after the wait: see launch.cuh)

    if (warp == kProducerWarp)
        tc_producer<true, tc_sep_p(NR), FUSED && tc_words_by_producer(NR)>(&tmK, &tmV, p, c);
    else if (warp == kVProducerWarp)
        tc_producer<false, tc_sep_p(NR), false>(&tmK, &tmV, p, c);
    else if (warp == kQkWarp) {
        if ((threadIdx.x & 31) == 0)
            tc_qk<NR>(p, c, tmem);
    } else if (warp == kPvWarp) {
        if ((threadIdx.x & 31) == 0)
            tc_pv<NR>(p, c, tmem);
    } else
        tc_softmax<NR, FUSED>(p, c, tmem);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Stages of 64 KiB that fit with the rest of the layout (0 if fewer than 2).
int umma_stages(int rows)
{
    int st = kTcMaxStages;
    while (st >= 2 && tc_smem_layout(rows, st, tc_sep_p(tc_nr(rows))).total > (uint32_t)kSmemLimit)
        --st;
    return st >= 2 ? st : 0;
}

uint32_t umma_smem_bytes(int rows, int stages) { return tc_smem_layout(rows, stages, tc_sep_p(tc_nr(rows))).total; }

template <int NR>
static cudaError_t launch_umma_t(const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p,
                                 uint32_t smem, cudaStream_t stream)
{
    auto kern = p.fused ? shkv_decode_umma_kernel<NR, true> : shkv_decode_umma_kernel<NR, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    return launch_pdl(kern, p.num_ctas, kTcThreads, smem, stream, tmK, tmV, p);
}

// tmK, tmV: 2-D maps of the pools (box of 64 columns x P rows, 128-byte swizzle).
cudaError_t launch_decode_umma(const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p, uint32_t smem,
                               cudaStream_t stream)
{
    switch (tc_nr(p.rows)) {
    case 16:
        return launch_umma_t<16>(tmK, tmV, p, smem, stream);
    case 32:
        return launch_umma_t<32>(tmK, tmV, p, smem, stream);
    case 48:
        return launch_umma_t<48>(tmK, tmV, p, smem, stream);
    case 64:
        return launch_umma_t<64>(tmK, tmV, p, smem, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace shkv
