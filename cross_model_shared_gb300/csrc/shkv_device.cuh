// shkv_device.cuh -- device-side building blocks for libshkv (sm_103a).
//
// Inline PTX wrappers for the Blackwell data-movement path (mbarrier, TMA
// tensor and bulk copies with L2 hints), the warp-level tensor-core path
// (ldmatrix, mma.sync m16n8k16 bf16, movmatrix) and bounded waits.  Every
// spin-wait here gives up after kWaitLimitNs of wall time, records
// SHKV_ERRF_TIMEOUT in the pool's error word and reports failure to the
// caller, which then skips work and drains its own in-flight copies; no
// kernel in this library can wait forever or trap.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "shkv.h"

namespace shkv {

// Tokens staged per pipeline slot (16 or 32).  A slot holds one or two
// row-blocks of min(page_size, kStageTokens) tokens of one KV head.
#ifndef SHKV_STAGE_TOKENS
#define SHKV_STAGE_TOKENS 32
#endif
constexpr int kStageTokens = SHKV_STAGE_TOKENS;
static_assert(kStageTokens == 16 || kStageTokens == 32, "stage is 16 or 32 tokens");
// Upper bound on pipeline slots per CTA (the ring also stops at the
// shared-memory limit).
#ifndef SHKV_MAX_STAGES
#define SHKV_MAX_STAGES 16
#endif
constexpr int kMaxStages = SHKV_MAX_STAGES;
// Consumer warps per row group, by number of row groups (1..4).  Fewer warps
// than ring slots keeps most of the ring in flight while warps compute.
#ifndef SHKV_WT_NT1
#define SHKV_WT_NT1 6          // rows per warp = 8 (R <= 8); the per-decoder-tails
                               // instantiation needs the extra warps, and the
                               // plain one takes the same count so that both
                               // combine a unit's stages in the same order
#endif
#ifndef SHKV_WT_NRG1
#define SHKV_WT_NRG1 3         // rows per warp = 16, one row group
#endif
#ifndef SHKV_WT_NRG2
#define SHKV_WT_NRG2 3
#endif
#ifndef SHKV_WT_NRG3
#define SHKV_WT_NRG3 2
#endif
#ifndef SHKV_WT_NRG4
#define SHKV_WT_NRG4 1
#endif
// Ring slots the producer arms and fills per iteration; each slot's copies
// are issued by four lanes, so one TMA instruction carries up to
// 4 * kStagesPerIssue copies.
#ifndef SHKV_STAGES_PER_ISSUE
#define SHKV_STAGES_PER_ISSUE 4
#endif
constexpr int kStagesPerIssue = SHKV_STAGES_PER_ISSUE;
// The producer takes page ids from a 32-entry block-table window that moves
// by 32 pages, so the pages of one issue pass (1 or 2 a stage) must divide
// 32: a pass that straddles the window's end would read wrapped entries.
static_assert(kStagesPerIssue == 1 || kStagesPerIssue == 2 || kStagesPerIssue == 4 || kStagesPerIssue == 8,
              "stages per issue: 1, 2, 4 or 8");
constexpr int kWtOfNrg[5] = {0, SHKV_WT_NRG1, SHKV_WT_NRG2, SHKV_WT_NRG3, SHKV_WT_NRG4};
// More than 16 stacked rows: use 8-row groups (no padding of R to 16) when
// set, else 16-row groups.  8-row groups take up to kNt1MultiWarps consumer
// warps in total.
#ifndef SHKV_R_ABOVE16_NT1
#define SHKV_R_ABOVE16_NT1 1
#endif
#ifndef SHKV_NT1_MULTI_WARPS
#define SHKV_NT1_MULTI_WARPS 10
#endif
constexpr int kNt1MultiWarps = SHKV_NT1_MULTI_WARPS;
constexpr int cmax(int a, int b) { return a > b ? a : b; }
// Largest blocks (consumer warps + one producer warp), per rows per warp.
constexpr int kMaxThreadsNT1 = 32 * (1 + cmax(SHKV_WT_NT1, kNt1MultiWarps));
constexpr int kMaxThreadsNT2 =
    32 * (1 + cmax(cmax(SHKV_WT_NRG1, 2 * SHKV_WT_NRG2), cmax(3 * SHKV_WT_NRG3, 4 * SHKV_WT_NRG4)));
// Largest number of consumer warps in one row group.
constexpr int kWtMax = cmax(cmax(cmax(SHKV_WT_NT1, kNt1MultiWarps / 2), SHKV_WT_NRG1),
                            cmax(cmax(SHKV_WT_NRG2, SHKV_WT_NRG3), SHKV_WT_NRG4));
// Stacked rows per KV head from which the automatic policy picks the tcgen05
// consumer (up to 64 rows); below it the mma.sync consumer runs.  A pool
// can name one consumer instead (shkv_pool_set_decode_consumer).
#ifndef SHKV_UMMA_MIN_ROWS
#define SHKV_UMMA_MIN_ROWS 16
#endif
constexpr int kUmmaMinRows = SHKV_UMMA_MIN_ROWS;
constexpr int kUmmaMaxRows = 64;
// Upper bound on persistent CTAs (one per SM).
constexpr int kMaxCtas = 256;
// Fixed cost of one (request, head) segment in the split plan, in page
// chunks: a CTA that crosses many short requests gets fewer chunks.
#ifndef SHKV_SEGMENT_COST_CHUNKS
#define SHKV_SEGMENT_COST_CHUNKS 16
#endif
constexpr int kSegmentCostChunks = SHKV_SEGMENT_COST_CHUNKS;
// Wall-clock limit for any single wait on an mbarrier.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
// Per ring slot, the producer publishes a word of valid pages + stage tag and,
// for fused tails, one page_info word per page of the stage (up to 8).
constexpr int kMetaWords = 16;
constexpr uint32_t kAllDecoders = 0xffu;
// Dynamic shared memory a CTA may use on sm_100-family parts.
constexpr int kSmemLimit = 232448;

struct DecodeParams {
    const __nv_bfloat16 *q;    // [B, N*Hq, D]
    __nv_bfloat16 *out;        // [B, N*Hq, D]
    float *lse_out;            // [B, N*Hq] or null
    const int32_t *block_table;
    // Per-decoder tails in one pass: when set, a request's unit of pages is
    // its shared pages followed by each decoder's tail pages (block_table is
    // that unit table), and page_info[b * max_pages + j] describes page j:
    // valid tokens (bits 0-7) and the decoder whose rows attend it (bits
    // 8-15, kAllDecoders for a shared page).
    const uint32_t *page_info;
    const int32_t *seq_lens;
    uint32_t *err;
    uint32_t *ws_count;        // [B*Hkv] arrival counters, zero between calls
    float *ws_lse;             // [2*C, R]
    float *ws_part;            // [2*C, R, D]
    int32_t batch, n_models, hq, hkv, group, rows;   // rows = R = N*G per KV head
    int32_t nrg, wt, rpad, stages;                   // row groups, token warps per group
    int32_t page_size, box_rows, max_pages, num_pages;
    int32_t num_ctas;
    int32_t split_producers;   // tcgen05 consumer: K and V copied by separate warps
    int64_t total_chunks;
    float scale_log2;
    int32_t fused;             // page_info is set (see above)
    int32_t cta_cut[kMaxCtas + 1];             // first chunk of each CTA; [num_ctas] = total
    int32_t page_prefix[SHKV_MAX_BATCH + 1];   // pages before each request
    uint8_t last_fill[SHKV_MAX_BATCH];         // tokens in each request's last page (1..P)
};

struct AppendParams {
    const uint4 *k_new, *v_new;    // [B, T, Hkv, D] bf16 as 16-byte vectors
    uint4 *k_pages, *v_pages;
    const int32_t *block_table;
    int32_t *seq_lens;
    uint32_t *err;
    int32_t batch, n_new, hkv, head_vecs, page_size, max_pages, num_pages, pad;
    int32_t old_len[SHKV_MAX_BATCH];
};

// ---------------------------------------------------------------------------
// shared-memory layout of the decode kernel (host and device agree on it)
// ---------------------------------------------------------------------------
struct DecodeSmem {
    uint32_t ring, stage_bytes, qbuf, qbuf_bytes, comb_o, comb_m, comb_l, bars, meta, misc, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// head_dim, rows per warp (8*NT), registers of O per lane, consumer warps, stages
__host__ __device__ inline DecodeSmem decode_smem_layout(int D, int rows_w, int nreg, int ncw,
                                                         int rpad, int stages)
{
    DecodeSmem s;
    s.stage_bytes = (uint32_t)(2 * kStageTokens * D * 2);
    s.ring = 0;
    s.qbuf = s.ring + (uint32_t)stages * s.stage_bytes;
    s.qbuf_bytes = (uint32_t)(rpad * D * 2);
    s.comb_o = align_up(s.qbuf + 2 * s.qbuf_bytes, 128);
    s.comb_m = s.comb_o + (uint32_t)(ncw * nreg * 32 * 4);
    s.comb_l = s.comb_m + (uint32_t)(ncw * rows_w * 4);
    s.bars = align_up(s.comb_l + (uint32_t)(ncw * rows_w * 4), 8);
    s.meta = s.bars + (uint32_t)((2 * stages + 4) * 8);
    s.misc = s.meta + (uint32_t)(stages * kMetaWords * 4);
    s.total = s.misc + 16 + 1024;   // + slack to align the base to 1024 bytes
    return s;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Programmatic dependent launch (kernels launched with
// cudaLaunchAttributeProgrammaticStreamSerialization).  A CTA waits for the
// previous kernel to complete, its memory visible, before it touches global
// memory, then lets the next kernel of the stream schedule its CTAs as SMs
// free up; both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait_prior() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity.  Returns false if the CTA's abort
// flag is raised or the wait runs over kWaitLimitNs (then the flag is raised
// and SHKV_ERRF_TIMEOUT recorded).  Per-thread; callers combine per warp.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t *abort_flag, uint32_t *err)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if ((it & 15u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1u;
            atomicOr(err, SHKV_ERRF_TIMEOUT);
            return false;
        }
    }
}

// Same, ignoring the abort flag: used only to drain copies this CTA issued.
__device__ __forceinline__ bool mbar_drain_bounded(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (globaltimer_ns() - t0 > kWaitLimitNs)
            return false;
    }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// 3-D tiled TMA load global -> shared at box origin (0, y, 0), completing on
// an mbarrier.
__device__ __forceinline__ void tma_load_3d_row(uint32_t dst, const CUtensorMap *tm, int y, uint32_t bar,
                                                uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(y), "r"(0), "r"(bar), "l"(policy)
        : "memory");
}

// 2-D tiled TMA load global -> shared at box origin (x, y); x * 2 bytes must
// be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int x, int y, uint32_t bar,
                                            uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// L2 prefetch of the box a tma_load_3d_row / tma_load_2d at the same
// coordinates would copy (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d_row(const CUtensorMap *tm, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(0), "r"(y), "r"(0)
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *tm, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Contiguous bulk copy global -> shared (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Device-scope acquire load (a split unit's arrival count).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *ptr)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *tm)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier among `nthreads` threads that also ORs a predicate over them.
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t nthreads, bool v)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)v), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float *c, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 bf16 matrix held one 32-bit pair per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// 2^x, the hardware approximation (MUFU.EX2); ex2(-inf) = +0.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void st_shared_zero16(uint32_t addr)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core) wrappers
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
//   K-major: rows of 128 bytes (64 bf16 along K), 8-row groups `sbo` apart.
//   MN-major: 128-byte rows run along M/N, `lbo` = byte distance between
//   64-element M/N blocks, `sbo` = byte distance between 8-row K groups.
__device__ __forceinline__ uint64_t umma_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;          // descriptor version
    d |= (uint64_t)2 << 61;          // 128-byte swizzle
    return d;
}

// Shared-memory matrix descriptor for an operand without swizzling (8-row x
// 16-byte core matrices; `lbo` and `sbo` are the byte strides between core
// matrices along K and along M/N).
__device__ __forceinline__ uint64_t umma_sdesc_noswz(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;          // descriptor version; layout type 0 = no swizzle
    return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, M x N, operand majorness.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] . B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_taddr, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_taddr),
                 "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrive on an mbarrier once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive 32-bit TMEM columns of this warp's 32 lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes, without the
// wait (tmem_wait_ld() completes it).
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld8_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8_nowait(uint32_t taddr, const uint32_t *r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t *r)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
                 "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
                 "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
                 "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace shkv
