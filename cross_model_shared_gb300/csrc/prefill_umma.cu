// prefill_umma.cu -- causal partial-prefill attention on the 5th-generation
// tensor cores (tcgen05 / TMEM), head dim 128.
//
// PrefillShare Sec. 3.3: on a prefix-cache hit the shared prefill module runs
// only on the n_new new tokens and extends the cached prefix.  Their K/V have
// been appended to the paged pool, so request b holds L_b tokens, the last
// n_new of them new; new token i sits at position L_b - n_new + i and
// attends every key at a position <= its own.
//
// A query tile is TPT = floor(128 / G) new tokens x the G query heads of one
// KV head: 128 MMA rows (row r = i * G + j), so every K/V page is read once
// for the whole group.  One CTA takes two consecutive tiles X = A, B of one
// (request, KV head) and streams 128-key stages of K and V through shared
// memory once for both (256 query rows per K/V byte).  Per stage and tile:
//   S_X[r, key]  = sum_d Q_X[r, d] K[key, d]      M = 128 rows, N = 128 keys
//   O_X[r, d]   += sum_key P_X[r, key] V[key, d]  M = 128 rows, N = 128 = D
// TMEM holds S_A, S_B, O_A, O_B (128 columns each).  A softmax thread owns one
// row of one tile (its TMEM lane): per stage it loads the row's 128 scores
// into registers, exponentiates them against its running maximum and writes P
// (bf16 pairs) over the first 64 columns of S, from where the PV product
// reads it.  Where every score of a warp's rows is visible and the running
// maxima are set, no stage maximum is taken; a row whose stage sum of P
// exceeds 2^16 (or is not finite) sends its warp through the exact path:
// mask, stage maximum, and a rescale of O and of the sum when the maximum
// moves by more than 2^kPRescaleLog2, then P again.  The
// two tiles keep the tensor core busy in turn: while one tile's softmax runs,
// the other tile's PV and next QK do.  Key stages past a tile's last position
// are skipped for that tile (and never loaded past the pair's last position);
// on the diagonal the causal mask is per element.
//
// Roles (384 threads): warps 0-3 softmax of tile A, warps 4-7 of tile B (row
// = TMEM lane), warp 8 QK issuer (its commit frees a K slot), warp 9 PV issuer
// (frees a V slot), warps 10 and 11 the K and V producers (TMA of page
// halves, one box per lane) on rings of their own.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "shkv_device.cuh"
#include "prefill.cuh"

namespace shkv {


namespace {

constexpr int kKT = 128;                 // keys per stage
constexpr int kPD = 128;                 // head dim
constexpr int kPHalves = kPD / 64;
constexpr int kPThreads = 384;
constexpr int kPQkWarp = 8;
constexpr int kPPvWarp = 9;
constexpr int kPKWarp = 10;
constexpr int kPVWarp = 11;
constexpr int kPGroupWarps = 4;          // softmax warps per tile
constexpr uint32_t kPTmemCols = 512;
constexpr float kPRescaleLog2 = 8.f;
#ifndef SHKV_PREFILL_K_SLOTS
#define SHKV_PREFILL_K_SLOTS 3
#endif
#ifndef SHKV_PREFILL_V_SLOTS
#define SHKV_PREFILL_V_SLOTS 2
#endif
// ring slots of 32 KB: a K slot is free once both tiles' QK have read it, a V
// slot only after both PVs, about one softmax later
constexpr int kKS = SHKV_PREFILL_K_SLOTS;
constexpr int kVS = SHKV_PREFILL_V_SLOTS;
constexpr int kPTilesPerCta = 2;
constexpr uint32_t kSlotBytes = (uint32_t)(kKT * kPD * 2);   // one operand of one stage: [half][128 keys][128 B]
constexpr uint32_t kQTileBytes = (uint32_t)(128 * kPD * 2);  // [half][128 rows][128 B]

// S of tile x (P over its first 64 columns), and O of tile x
__device__ __forceinline__ uint32_t col_s(int x) { return (uint32_t)(x * 128); }
__device__ __forceinline__ uint32_t col_o(int x) { return (uint32_t)(256 + x * 128); }

// Registers per thread after the split of the launch's 168 (setmaxnreg): the
// two softmax warpgroups hold a whole 128-score row in registers; the MMA
// issuers and the producers need few.  224 * 256 + 56 * 128 = 168 * 384.
constexpr uint32_t kPSoftmaxRegs = 224;
constexpr uint32_t kPOtherRegs = 56;
static_assert(kPSoftmaxRegs * 256 + kPOtherRegs * 128 == 168 * kPThreads, "register split");

__device__ __forceinline__ void setmaxnreg_inc(void) { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPSoftmaxRegs)); }
__device__ __forceinline__ void setmaxnreg_dec(void) { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPOtherRegs)); }

// max of three (one instruction on sm_100 and later)
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float y;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
    return y;
}

// D[tmem] (+)= A[tmem] . B[smem]^T, issued by one thread: A is 128 lanes
// (rows) x K columns of packed bf16 pairs, the lower half the lower k.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_taddr),
                 "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Bounded wait that sleeps on the barrier instead of spinning: each try_wait
// suspends the thread until the phase completes or ~20 us pass, so waiting
// warps leave the issue slots to the softmax warps of their SM sub-partition.
// Gives up like mbar_wait_bounded (abort flag, or SHKV_ERRF_TIMEOUT after
// kWaitLimitNs).
__device__ __forceinline__ bool pf_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

__device__ bool pf_wait(uint32_t bar, uint32_t parity, volatile uint32_t *abort_flag, uint32_t *err)
{
    if (pf_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (pf_try_wait(bar, parity))
            return true;
        if (*abort_flag)
            return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1u;
            atomicOr(err, SHKV_ERRF_TIMEOUT);
            return false;
        }
    }
}

struct PfSmem {
    uint32_t qtile, kring, vring, bars, misc, tslot, total;
};

// the two Q tiles [tile][half][128 rows][128 B], the K ring and the V ring
// (slots [half][128 keys][128 B]; all 128-byte swizzled), then the barriers:
// full_k[KS], empty_k[KS], full_v[VS], empty_v[VS], s_full[tile],
// p_full[tile], pv_done[tile], fin, q_ready.  A tile's S is rewritten by its
// next QK only after its PV has read the P over it, so none of the per-tile
// barriers can run two phases ahead of a waiter.
__host__ __device__ inline PfSmem pf_layout()
{
    PfSmem u;
    u.qtile = 0;
    u.kring = u.qtile + (uint32_t)kPTilesPerCta * kQTileBytes;
    u.vring = u.kring + (uint32_t)kKS * kSlotBytes;
    u.bars = u.vring + (uint32_t)kVS * kSlotBytes;
    u.misc = u.bars + (uint32_t)((2 * (kKS + kVS) + 8) * 8);
    u.tslot = u.misc + 8;
    u.total = u.misc + 16 + 1024;
    return u;
}

struct PfCtx {
    uint8_t *smem;
    uint32_t base;
    PfSmem lay;
    volatile uint32_t *abort_flag;
};

__device__ __forceinline__ uint32_t pbar(const PfCtx &c, int i) { return c.base + c.lay.bars + 8u * i; }
__device__ __forceinline__ uint32_t pf_full(const PfCtx &c, bool v, int s)
{
    return pbar(c, v ? 2 * kKS + s : s);
}
__device__ __forceinline__ uint32_t pf_empty(const PfCtx &c, bool v, int s)
{
    return pbar(c, v ? 2 * kKS + kVS + s : kKS + s);
}
constexpr int kPTileBar0 = 2 * (kKS + kVS);
__device__ __forceinline__ uint32_t pf_sfull(const PfCtx &c, int x) { return pbar(c, kPTileBar0 + x); }
__device__ __forceinline__ uint32_t pf_pfull(const PfCtx &c, int x) { return pbar(c, kPTileBar0 + 2 + x); }
__device__ __forceinline__ uint32_t pf_pvdone(const PfCtx &c, int x) { return pbar(c, kPTileBar0 + 4 + x); }
__device__ __forceinline__ uint32_t pf_fin(const PfCtx &c) { return pbar(c, kPTileBar0 + 6); }
// both query tiles are in shared memory (one arrival per softmax warp)
__device__ __forceinline__ uint32_t pf_qready(const PfCtx &c) { return pbar(c, kPTileBar0 + 7); }
__device__ __forceinline__ uint32_t pf_kslot(const PfCtx &c, int s) { return c.base + c.lay.kring + (uint32_t)s * kSlotBytes; }
__device__ __forceinline__ uint32_t pf_vslot(const PfCtx &c, int s) { return c.base + c.lay.vring + (uint32_t)s * kSlotBytes; }
// parity of stage k's use of a ring of n slots
__device__ __forceinline__ uint32_t ring_par(int k, int n) { return (uint32_t)((k / n) & 1); }

// the pair of tiles this CTA owns
struct Tile {
    int b, g;
    int L, prefix;               // request length (with the new tokens), cached tokens before them
    int i0[2], ntok[2];          // first new token and new tokens of tiles A and B (B may be empty)
    int nst[2];                  // key stages each tile attends: keys 0 .. its last position
    int nst_all;                 // stages loaded: the larger of the two
};

// CTAs are dispatched roughly in index order, so the index runs over the
// longest work first (requests by length, then each request's tile pairs from
// the last, which attends the most keys): the short pairs fill the last wave.
__device__ __forceinline__ Tile pf_tile(const PrefillParams &p)
{
    Tile t;
    const int pairs = (p.tiles + kPTilesPerCta - 1) / kPTilesPerCta;
    int idx = blockIdx.x;
    const int tp = pairs - 1 - idx % pairs;
    idx /= pairs;
    t.g = idx % p.hkv;
    t.b = p.order[idx / p.hkv];
    t.L = p.lens[t.b];
    t.prefix = t.L - p.n_new;
#pragma unroll
    for (int x = 0; x < kPTilesPerCta; ++x) {
        t.i0[x] = (kPTilesPerCta * tp + x) * p.tpt;
        t.ntok[x] = max(0, min(p.tpt, p.n_new - t.i0[x]));
        t.nst[x] = t.ntok[x] > 0 ? (t.prefix + t.i0[x] + t.ntok[x] - 1) / kKT + 1 : 0;
    }
    t.nst_all = max(t.nst[0], t.nst[1]);
    return t;
}

// ---------------------------------------------------------------------------
// producers: stage k = keys [128k, 128k + 128), 128/P pages; one warp copies
// the K halves of the pages into the K ring, another the V halves into the V
// ring (one box per lane).  A page whose block-table entry lies outside the
// pool is not copied (the V producer flags it); the softmax masks its keys.
// ---------------------------------------------------------------------------
template <bool kIsV>
__device__ void pf_producer(const CUtensorMap *tm, const PrefillParams &p, const PfCtx &c, const Tile &t)
{
    constexpr int S = kIsV ? kVS : kKS;
    const int lane = threadIdx.x & 31;
    const int P = p.page_size;
    const int RB = kKT / P;
    const int my_h = lane / RB, my_rb = lane % RB;
    const bool copier = lane < kPHalves * RB;
    const uint32_t page_bytes = kPHalves * (uint32_t)P * 128u;
    const uint64_t pol = l2_evict_first_policy();
    if (lane == 0) {
        prefetch_tensormap(tm);
        if (kIsV && __ldg(p.seq_lens + t.b) != t.L)
            atomicOr(p.err, SHKV_ERRF_SEQ_LEN);
    }
    const int npages = (t.L + P - 1) / P;
    const int32_t *btrow = p.block_table + (int64_t)t.b * p.max_pages;
    bool alive = true;
    int last_issued = -1;
    // page ids are read one stage ahead
    int nxt_id = (copier && my_rb < npages) ? __ldg(btrow + my_rb) : -1;
    for (int k = 0; k < t.nst_all; ++k) {
        const int slot = k % S;
        const int pg = k * RB + my_rb;
        const int my_id = nxt_id;
        {
            const int pgn = (k + 1) * RB + my_rb;
            nxt_id = (k + 1 < t.nst_all && copier && pgn < npages) ? __ldg(btrow + pgn) : -1;
        }
        bool ok = true;
        if (alive && lane == 0)
            ok = pf_wait(pf_empty(c, kIsV, slot), ring_par(k, S) ^ 1u, c.abort_flag, p.err);
        alive = alive && __all_sync(0xffffffffu, ok);
        const bool my_valid = copier && pg < npages && my_id >= 0 && my_id < p.num_pages;
        const uint32_t mask = __ballot_sync(0xffffffffu, my_valid) & ((1u << RB) - 1u);
        if (alive && lane == 0) {
            if (kIsV)
                for (int rb = 0; rb < RB; ++rb)
                    if (!((mask >> rb) & 1u) && k * RB + rb < npages)
                        atomicOr(p.err, SHKV_ERRF_PAGE_OOB);
            mbar_arrive_expect_tx(pf_full(c, kIsV, slot), (uint32_t)__popc(mask) * page_bytes);
        }
        __syncwarp();
        if (alive && my_valid) {
            const uint32_t dst = (kIsV ? pf_vslot(c, slot) : pf_kslot(c, slot)) + (uint32_t)my_h * (kKT * 128) +
                                 (uint32_t)my_rb * (uint32_t)P * 128u;
            tma_load_2d(dst, tm, my_h * 64, (my_id * p.hkv + t.g) * P, pf_full(c, kIsV, slot), pol);
        }
        if (alive)
            last_issued = k;
        __syncwarp();
    }
    if (!alive && lane == 0)
        for (int k = last_issued - S + 1; k <= last_issued; ++k)
            if (k >= 0)
                mbar_drain_bounded(pf_full(c, kIsV, k % S), ring_par(k, S));
}

// ---------------------------------------------------------------------------
// MMA issuers
// ---------------------------------------------------------------------------
// S_X = Q_X K^T (N = 128 keys) for each tile that attends stage k, once
// PV_X(k-1) has read the P written over S_X.  The descriptors are built from
// one base each by adding (byte offset >> 4) to the 14-bit address field,
// which shared addresses below 256 KB never carry out of.
__device__ void pf_qk(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem)
{
    const uint32_t idesc = umma_idesc_bf16(128, kKT, false, false);
    const uint64_t qd0 = umma_sdesc_sw128(c.base + c.lay.qtile, 16u, 1024u);
    const uint64_t kd0 = umma_sdesc_sw128(pf_kslot(c, 0), 16u, 1024u);
    bool alive = pf_wait(pf_qready(c), 0u, c.abort_flag, p.err);
    for (int k = 0; k < t.nst_all; ++k) {
        const int slot = k % kKS;
        const uint64_t kd = kd0 + (((uint32_t)slot * kSlotBytes) >> 4);
        if (alive)
            alive = pf_wait(pf_full(c, false, slot), ring_par(k, kKS), c.abort_flag, p.err);
#pragma unroll
        for (int x = 0; x < kPTilesPerCta; ++x) {
            if (k >= t.nst[x])
                continue;
            if (alive && k >= 1)
                alive = pf_wait(pf_pvdone(c, x), (uint32_t)((k - 1) & 1), c.abort_flag, p.err);
            if (alive) {
                tc_fence_after();
                const uint32_t d = tmem + col_s(x);
                const uint64_t qd = qd0 + (((uint32_t)x * kQTileBytes) >> 4);
#pragma unroll
                for (int i = 0; i < kPHalves * 4; ++i) {
                    const uint32_t off = (uint32_t)((i >> 2) * 128 * 128 + (i & 3) * 32) >> 4;
                    umma_bf16(d, qd + off, kd + off, idesc, i ? 1u : 0u);
                }
            }
            umma_commit(pf_sfull(c, x));
        }
        umma_commit(pf_empty(c, false, slot));
    }
    umma_commit(pf_fin(c));
    mbar_drain_bounded(pf_fin(c), 0u);
}

// O_X += P_X V; P_X from TMEM (over S_X), V MN-major in the V slot.  PV_A(k)
// waits for tile A's softmax, which also cleared the stage's unusable V rows
// for both tiles (tile B's alone once A no longer attends the stage).
__device__ void pf_pv(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem)
{
    const uint32_t idesc = umma_idesc_bf16(128, kPD, false, true);
    const uint64_t vd0 = umma_sdesc_sw128(pf_vslot(c, 0), (uint32_t)(kKT * 128), 1024u);
    bool alive = true;
    for (int k = 0; k < t.nst_all; ++k) {
        const int slot = k % kVS;
        const uint64_t vd = vd0 + (((uint32_t)slot * kSlotBytes) >> 4);
        if (alive)
            alive = pf_wait(pf_full(c, true, slot), ring_par(k, kVS), c.abort_flag, p.err);
#pragma unroll
        for (int x = 0; x < kPTilesPerCta; ++x) {
            if (k >= t.nst[x])
                continue;
            if (alive)
                alive = pf_wait(pf_pfull(c, x), (uint32_t)(k & 1), c.abort_flag, p.err);
            if (alive) {
                tc_fence_after();
                const uint32_t d = tmem + col_o(x);
                const uint32_t a = tmem + col_s(x);
#pragma unroll
                for (int ks = 0; ks < kKT / 16; ++ks)
                    umma_bf16_ts(d, a + (uint32_t)(ks * 8), vd + (uint64_t)((ks * 2048u) >> 4), idesc,
                                 (k == 0 && ks == 0) ? 0u : 1u);
            }
            umma_commit(pf_pvdone(c, x));
        }
        umma_commit(pf_empty(c, true, slot));
    }
    umma_commit(pf_fin(c));
    mbar_drain_bounded(pf_fin(c), 0u);
}

// ---------------------------------------------------------------------------
// softmax warps of tile x: thread r = MMA row r = (new token i0 + r / G, head r % G)
// ---------------------------------------------------------------------------
__device__ void pf_softmax(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem, int x,
                           float &m_out, float &l_out, bool &alive_out)
{
    const int r = threadIdx.x - x * 128;
    const int lane = r & 31, warp = r >> 5;
    const int ti = r / p.group;
    const bool row_ok = ti < t.ntok[x];
    const int pos = t.prefix + t.i0[x] + ti;             // this row's position (keys 0 .. pos)
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint32_t orow = tmem + lane_base + col_o(x);
    const uint32_t srow = tmem + lane_base + col_s(x);
    const int P = p.page_size;
    const int log2P = 31 - __clz(P);
    const int RB = kKT / P;
    const uint32_t all_pages = (1u << RB) - 1u;
    const int npages = (t.L + P - 1) / P;
    const int32_t *btrow = p.block_table + (int64_t)t.b * p.max_pages;
    const float sl2 = p.scale_log2;
    float m_use = -INFINITY, lsum = 0.f;
    bool alive = true;
    // the softmax warps poll their barriers (measured faster than sleeping
    // on them, which the issuers and producers do): their waits sit on the
    // tile's chain QK -> softmax -> PV
    auto wait = [&](uint32_t bar, uint32_t parity) {
        bool ok = false;
        if (alive)
            ok = mbar_wait_bounded(bar, parity, c.abort_flag, p.err);
        alive = __all_sync(0xffffffffu, ok) && alive;
        return alive;
    };
    // the pages the producers copy: lane l < RB reads the block-table entry of
    // the stage's page l (one stage ahead) and applies the producers' test
    int nxt_id = (lane < RB && lane < npages) ? __ldg(btrow + lane) : -1;
    for (int k = 0; k < t.nst[x]; ++k) {
        const int key0 = k * kKT;
        const int my_id = nxt_id;
        {
            const int pgn = (k + 1) * RB + lane;
            nxt_id = (k + 1 < t.nst[x] && lane < RB && pgn < npages) ? __ldg(btrow + pgn) : -1;
        }
        const bool page_ok = lane < RB && k * RB + lane < npages && my_id >= 0 && my_id < p.num_pages;
        const uint32_t pmask = __ballot_sync(0xffffffffu, page_ok) & all_pages;
        // keys this row may see: [key0, key0 + nvis), on pages that were copied
        const int nvis = row_ok ? min(kKT, pos - key0 + 1) : 0;
        // no mask below the diagonal; padding rows (no token) need none either:
        // their scores only reach their own row of O, which is not stored
        const bool dense = pmask == all_pages && (nvis == kKT || !row_ok);
        wait(pf_sfull(c, x), (uint32_t)(k & 1));
        if (alive)
            tc_fence_after();
        // this row's 128 scores into registers, masked (-inf where invisible)
        uint32_t sv[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            tmem_ld32_nowait(srow + (uint32_t)(q * 32), sv[q]);
        tmem_wait_ld();
        // P = 2^(s * scale_log2 - mu) as bf16 pairs over columns 0 .. 63 of S
        // (the scores are in registers); returns the row's sum of P.  The
        // scaling and the sums run on packed fp32 pairs (one issue slot for
        // two results), the exponentials on the SFU.
        auto exp_store = [&](float mu) -> float {
            const float2 sl2x2 = make_float2(sl2, sl2), nmu2 = make_float2(-mu, -mu);
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 xe = __ffma2_rn(
                        make_float2(__uint_as_float(sv[q][2 * e]), __uint_as_float(sv[q][2 * e + 1])), sl2x2, nmu2);
                    const float2 pe = make_float2(ex2_approx(xe.x), ex2_approx(xe.y));
                    acc[e & 3] = __fadd2_rn(acc[e & 3], pe);
                    pk[e] = pack_bf16x2(pe.x, pe.y);
                }
                tmem_st16_nowait(srow + (uint32_t)(q * 16), pk);
            }
            const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
            return (a01.x + a01.y) + (a23.x + a23.y);
        };
        // Common case: every score of the warp's rows is visible and the
        // running maxima are set, so P is taken against them without this
        // stage's maximum.  A row whose stage sum exceeds 2^16 (some weight
        // above 2^9 against its running maximum) or is not finite sends the
        // warp through the exact path below, which rewrites P.
        float part = 0.f;
        bool fast = __all_sync(0xffffffffu, dense && alive && m_use != -INFINITY);
        if (fast) {
            part = exp_store(m_use);
            if (__any_sync(0xffffffffu, !(part <= 65536.f))) {
                tmem_wait_st();
                fast = false;
            }
        }
        if (!fast) {
            if (!dense || !alive) {
    #pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // bit e: column 32q + e is visible (before this row's end, on a copied page)
                    const int n = alive ? min(max(nvis - q * 32, 0), 32) : 0;
                    uint32_t vis = n >= 32 ? 0xffffffffu : ((1u << n) - 1u);
                    uint32_t pages = 0u;
                    for (int pg = 0; pg < 32 / P; ++pg)
                        if ((pmask >> (q * (32 / P) + pg)) & 1u)
                            pages |= (P >= 32 ? 0xffffffffu : ((1u << P) - 1u)) << (pg * P);
                    vis &= pages;
    #pragma unroll
                    for (int e = 0; e < 32; ++e)
                        sv[q][e] = ((vis >> e) & 1u) ? sv[q][e] : __float_as_uint(-INFINITY);
                }
            }
            float cm;
            {
                float a = -INFINITY, b = -INFINITY, d = -INFINITY, e4 = -INFINITY;
    #pragma unroll
                for (int q = 0; q < 4; ++q)
    #pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        a = max3f(a, __uint_as_float(sv[q][e]), __uint_as_float(sv[q][e + 1]));
                        b = max3f(b, __uint_as_float(sv[q][e + 2]), __uint_as_float(sv[q][e + 3]));
                        d = max3f(d, __uint_as_float(sv[q][e + 4]), __uint_as_float(sv[q][e + 5]));
                        e4 = max3f(e4, __uint_as_float(sv[q][e + 6]), __uint_as_float(sv[q][e + 7]));
                    }
                cm = max3f(a, b, fmaxf(d, e4));
            }
            // the running maximum moves only by more than 2^kPRescaleLog2 (or when
            // it is first set; O and the sum are still zero then)
            const float mt = cm * sl2;                                // sl2 > 0; -inf if nothing is visible
            const bool first = m_use == -INFINITY && mt != -INFINITY;
            const bool need = alive && m_use != -INFINITY && mt > m_use + kPRescaleLog2;
            if (first)
                m_use = mt;
            if (__any_sync(0xffffffffu, need)) {
                // tcgen05.ld/st are warp-wide: lanes that keep their maximum scale by 1
                const float alpha = need ? ex2_approx(m_use - mt) : 1.f;
                if (k >= 1) {
                    wait(pf_pvdone(c, x), (uint32_t)((k - 1) & 1));
                    if (alive) {
                        tc_fence_after();
    #pragma unroll 1
                        for (int c32 = 0; c32 < kPD / 32; ++c32) {
                            uint32_t ov[32];
                            tmem_ld32(orow + (uint32_t)(c32 * 32), ov);
    #pragma unroll
                            for (int e = 0; e < 32; ++e)
                                ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                            tmem_st32(orow + (uint32_t)(c32 * 32), ov);
                        }
                    }
                }
                if (need) {
                    lsum *= alpha;
                    m_use = mt;
                }
            }
            part = exp_store(m_use == -INFINITY ? 0.f : m_use);
        }
        lsum += part;
        tmem_wait_st();
        tc_fence_before();
        // V rows of keys that no row may use in this stage (past the request's
        // end, or on a skipped page) may hold stale or non-finite bits: zero
        // them (thread r takes key row r) once V has landed.  Tile A does it
        // while it attends the stage, tile B after that.
        const bool zero_stage = key0 + kKT > t.L || pmask != all_pages;
        if (zero_stage && (x == 0 || k >= t.nst[0])) {
            wait(pf_full(c, true, k % kVS), ring_par(k, kVS));
            const int key = key0 + r;
            const bool zero_mine = alive && !(key < t.L && ((pmask >> (r >> log2P)) & 1u));
            if (__any_sync(0xffffffffu, zero_mine)) {
                if (zero_mine) {
                    const uint32_t vrow = pf_vslot(c, k % kVS) + (uint32_t)r * 128u;
#pragma unroll
                    for (int hh = 0; hh < kPHalves; ++hh)
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch)
                            st_shared_zero16(vrow + (uint32_t)(hh * kKT * 128 + ch * 16));
                }
                fence_proxy_async_smem();
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(pf_pfull(c, x));
    }
    m_out = m_use;
    l_out = lsum;
    alive_out = alive;
}

// ---------------------------------------------------------------------------
// epilogue: this row of O_x, normalised, and its log-sum-exp
// ---------------------------------------------------------------------------
__device__ void pf_epilogue(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem, int x,
                            float m_use, float lsum, bool alive)
{
    const int r = threadIdx.x - x * 128;
    const int warp = r >> 5;
    const int ti = r / p.group, tj = r - (r / p.group) * p.group;
    const bool row_ok = ti < t.ntok[x];
    const uint32_t orow = tmem + ((uint32_t)(warp * 32) << 16) + col_o(x);
    const int last = t.nst[x] - 1;
    if (last < 0)
        return;                                  // tile B of an odd tile count: no rows
    bool ok = alive && pf_wait(pf_pvdone(c, x), (uint32_t)(last & 1), c.abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok)
        return;
    tc_fence_after();
    const float inv = lsum > 0.f ? __frcp_rn(lsum) : 0.f;
    const int64_t row = ((int64_t)t.b * p.n_new + t.i0[x] + ti) * p.hq + (int64_t)t.g * p.group + tj;
#pragma unroll 1
    for (int c32 = 0; c32 < kPD / 32; ++c32) {
        uint32_t ov[32];
        tmem_ld32(orow + (uint32_t)(c32 * 32), ov);
        if (row_ok) {
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * kPD + c32 * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 2 * e]) * inv,
                                       __uint_as_float(ov[q4 * 8 + 2 * e + 1]) * inv);
                dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    }
    tc_fence_before();
    if (row_ok && p.lse_out)
        p.lse_out[row] = lsum > 0.f ? (m_use + log2f(lsum)) * 0.6931471805599453f : -INFINITY;
}

}  // namespace

__global__ void __launch_bounds__(kPThreads, 1)
    shkv_prefill_umma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                             const __grid_constant__ PrefillParams p)
{
    extern __shared__ uint8_t smem_raw[];
    PfCtx c;
    {
        const uint32_t raw = smem_u32(smem_raw);
        const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
        c.smem = smem_raw + pad;
        c.base = raw + pad;
    }
    c.lay = pf_layout();
    c.abort_flag = reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.misc);
    const Tile t = pf_tile(p);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kKS; ++s) {
            mbar_init(pf_full(c, false, s), 1);
            mbar_init(pf_empty(c, false, s), 1);
        }
        for (int s = 0; s < kVS; ++s) {
            mbar_init(pf_full(c, true, s), 1);
            mbar_init(pf_empty(c, true, s), 1);
        }
        for (int x = 0; x < kPTilesPerCta; ++x) {
            mbar_init(pf_sfull(c, x), 1);
            mbar_init(pf_pfull(c, x), kPGroupWarps);
            mbar_init(pf_pvdone(c, x), 1);
        }
        mbar_init(pf_fin(c), 2);
        mbar_init(pf_qready(c), kPTilesPerCta * kPGroupWarps);
        *c.abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp == 0)
        tmem_alloc(c.base + c.lay.tslot, kPTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.tslot);

    if (warp >= kPQkWarp) {
        // warpgroup 2: the MMA issuers and the producers give registers up
        setmaxnreg_dec();
        if (warp == kPKWarp)
            pf_producer<false>(&tmK, p, c, t);
        else if (warp == kPVWarp)
            pf_producer<true>(&tmV, p, c, t);
        else if (warp == kPQkWarp) {
            if ((threadIdx.x & 31) == 0)
                pf_qk(p, c, t, tmem);
        } else if (warp == kPPvWarp) {
            if ((threadIdx.x & 31) == 0)
                pf_pv(p, c, t, tmem);
        }
    } else {
        // warpgroups 0 and 1: the softmax of tiles A and B takes them
        setmaxnreg_inc();
        // this thread's query row into its tile's swizzled K-major Q tile
        // (padding rows zero), after the CTA barrier so that the producers'
        // first copies are already on their way
        const int x = warp / kPGroupWarps;
        {
            const int r = threadIdx.x - x * 128;
            const int ti = r / p.group, tj = r - (r / p.group) * p.group;
            const bool row_ok = ti < t.ntok[x];
            const uint4 *src = reinterpret_cast<const uint4 *>(
                p.q + (((int64_t)t.b * p.n_new + t.i0[x] + ti) * p.hq + (int64_t)t.g * p.group + tj) * kPD);
            const uint32_t qtile = c.lay.qtile + (uint32_t)x * kQTileBytes;
#pragma unroll
            for (int ch = 0; ch < kPD / 8; ++ch) {
                const uint4 v = row_ok ? __ldg(src + ch) : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t off = (uint32_t)(ch >> 3) * (128u * 128u) + (uint32_t)r * 128u +
                                     (uint32_t)(((ch & 7) ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(c.smem + qtile + off) = v;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if ((threadIdx.x & 31) == 0)
                mbar_arrive(pf_qready(c));
        }
        float m_use, lsum;
        bool alive;
        pf_softmax(p, c, t, tmem, x, m_use, lsum, alive);
        pf_epilogue(p, c, t, tmem, x, m_use, lsum, alive);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(tmem, kPTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int prefill_tiles_per_cta() { return kPTilesPerCta; }

uint32_t prefill_smem_bytes() { return pf_layout().total; }

// tmK, tmV: 2-D maps of the pools (box of 64 columns x P rows, 128-byte swizzle).
cudaError_t launch_prefill_umma(const CUtensorMap &tmK, const CUtensorMap &tmV, const PrefillParams &p, uint32_t smem,
                                int grid, cudaStream_t stream)
{
    // The setmaxnreg split hands out exactly the registers the CTA is launched
    // with (168 a thread): a build with another count is refused rather than
    // launched, since its setmaxnreg.inc could wait for registers forever.
    static int num_regs = -1;
    if (num_regs < 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, shkv_prefill_umma_kernel);
        if (e != cudaSuccess)
            return e;
        num_regs = fa.numRegs;
    }
    if ((uint32_t)num_regs * kPThreads != kPSoftmaxRegs * 256 + kPOtherRegs * 128)
        return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(shkv_prefill_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    shkv_prefill_umma_kernel<<<grid, kPThreads, smem, stream>>>(tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace shkv
