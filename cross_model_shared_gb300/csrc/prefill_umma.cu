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
// (request, KV head) and streams 64-key stages of K/V through shared memory
// once for both (256 query rows per K/V byte).  Per stage and tile:
//   S_X[r, key]  = sum_d Q_X[r, d] K[key, d]      M = 128 rows, N = 64 keys
//   O_X[r, d]   += sum_key P_X[r, key] V[key, d]  M = 128 rows, N = 128 = D
// TMEM holds two S buffers per tile (64 columns each) and O_A, O_B (128
// each), so QK of the next stage runs while the softmax works on this one.  A
// softmax thread owns one row of one tile (its TMEM lane): it loads its 64
// scores into registers, takes their maximum, exponentiates them against its
// running maximum and writes P (bf16 pairs) over the first 32 columns of the
// S buffer, from where the PV product reads it.  The running maximum moves
// only when the stage maximum exceeds it by more than 2^kPRescaleLog2; the
// thread then rescales its row of O first.  Key stages past a tile's last
// position are skipped for that tile (and never loaded past the pair's last
// position); on the diagonal the causal mask is per element.
//
// Roles (384 threads): warps 0-3 softmax of tile A, warps 4-7 of tile B (row
// = TMEM lane), warp 8 QK issuer (its commit frees the K half of a ring slot),
// warp 9 PV issuer (frees the V half), warps 10 and 11 the K and V producers
// (TMA of page halves, one box per lane).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "shkv_device.cuh"
#include "prefill.cuh"

namespace shkv {


namespace {

constexpr int kKT = 64;                  // keys per stage
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
constexpr int kPStages = 4;              // ring slots of 32 KB
constexpr int kPTilesPerCta = 2;

// S buffer b of tile x (P over its first 32 columns), and O of tile x
__device__ __forceinline__ uint32_t col_s(int x, int b) { return (uint32_t)(x * 128 + b * 64); }
__device__ __forceinline__ uint32_t col_o(int x) { return (uint32_t)(256 + x * 128); }

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
    uint32_t ring, stage_bytes, qtile, bars, meta, misc, tslot, total;
};

// ring slots of [K | V][half][64 keys][128 B], then the two Q tiles
// [tile][half][128 rows][128 B] (all 128-byte swizzled), then the barriers:
// full_k[S], full_v[S], empty_k[S], empty_v[S], s_full[tile][buf], p_full[tile][buf],
// pv_done[tile][buf], fin, q_ready.  Everything a tile's softmax hands to the MMA
// issuers is per S buffer: a softmax group may finish stage k+1 before the
// PV issuer has waited for stage k, but not stage k+2 (its scores need PV(k)).
__host__ __device__ inline PfSmem pf_layout()
{
    PfSmem u;
    u.stage_bytes = (uint32_t)(2 * kKT * kPD * 2);
    u.ring = 0;
    u.qtile = (uint32_t)kPStages * u.stage_bytes;
    u.bars = u.qtile + (uint32_t)(kPTilesPerCta * kPHalves * 128 * 128);
    u.meta = u.bars + (uint32_t)((4 * kPStages + 14) * 8);
    u.misc = u.meta + (uint32_t)(kPStages * 4);
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
__device__ __forceinline__ uint32_t pf_full(const PfCtx &c, bool v, int s) { return pbar(c, (v ? kPStages : 0) + s); }
__device__ __forceinline__ uint32_t pf_empty(const PfCtx &c, bool v, int s)
{
    return pbar(c, (v ? 3 : 2) * kPStages + s);
}
__device__ __forceinline__ uint32_t pf_sfull(const PfCtx &c, int x, int b) { return pbar(c, 4 * kPStages + 2 * x + b); }
__device__ __forceinline__ uint32_t pf_pfull(const PfCtx &c, int x, int b) { return pbar(c, 4 * kPStages + 4 + 2 * x + b); }
__device__ __forceinline__ uint32_t pf_pvdone(const PfCtx &c, int x, int b)
{
    return pbar(c, 4 * kPStages + 8 + 2 * x + b);
}
__device__ __forceinline__ uint32_t pf_fin(const PfCtx &c) { return pbar(c, 4 * kPStages + 12); }
// both query tiles are in shared memory (one arrival per softmax warp)
__device__ __forceinline__ uint32_t pf_qready(const PfCtx &c) { return pbar(c, 4 * kPStages + 13); }
__device__ __forceinline__ uint32_t pf_slot(const PfCtx &c, int s)
{
    return c.base + c.lay.ring + (uint32_t)s * c.lay.stage_bytes;
}
__device__ __forceinline__ uint32_t ring_par(int k) { return (uint32_t)((k / kPStages) & 1); }

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
// producers: stage k = keys [64k, 64k + 64), 64/P pages; one warp copies
// the K halves of the pages, another the V halves (one box per lane).  The V
// producer records which pages it copied in the slot's word (a V half is
// released only after both tiles' softmax of its stage have read the word).
// ---------------------------------------------------------------------------
template <bool kIsV>
__device__ void pf_producer(const CUtensorMap *tm, const PrefillParams &p, const PfCtx &c, const Tile &t)
{
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
        const int slot = k % kPStages;
        const int pg = (k * kKT) / P + my_rb;
        const int my_id = nxt_id;
        {
            const int pgn = ((k + 1) * kKT) / P + my_rb;
            nxt_id = (k + 1 < t.nst_all && copier && pgn < npages) ? __ldg(btrow + pgn) : -1;
        }
        bool ok = true;
        if (alive && lane == 0)
            ok = pf_wait(pf_empty(c, kIsV, slot), ring_par(k) ^ 1u, c.abort_flag, p.err);
        alive = alive && __all_sync(0xffffffffu, ok);
        const bool my_valid = copier && pg < npages && my_id >= 0 && my_id < p.num_pages;
        const uint32_t mask = __ballot_sync(0xffffffffu, my_valid) & ((1u << RB) - 1u);
        if (alive && lane == 0) {
            if (kIsV) {
                for (int rb = 0; rb < RB; ++rb)
                    if (!((mask >> rb) & 1u) && (k * kKT) / P + rb < npages)
                        atomicOr(p.err, SHKV_ERRF_PAGE_OOB);
                reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.meta)[slot] = mask | ((uint32_t)k << 8);
            }
            mbar_arrive_expect_tx(pf_full(c, kIsV, slot), (uint32_t)__popc(mask) * page_bytes);
        }
        __syncwarp();
        if (alive && my_valid) {
            const uint32_t dst = pf_slot(c, slot) + (kIsV ? (uint32_t)(kKT * kPD * 2) : 0u) +
                                 (uint32_t)my_h * (kKT * 128) + (uint32_t)my_rb * (uint32_t)P * 128u;
            tma_load_2d(dst, tm, my_h * 64, (my_id * p.hkv + t.g) * P, pf_full(c, kIsV, slot), pol);
        }
        if (alive)
            last_issued = k;
        __syncwarp();
    }
    if (!alive && lane == 0)
        for (int k = last_issued - kPStages + 1; k <= last_issued; ++k)
            if (k >= 0)
                mbar_drain_bounded(pf_full(c, kIsV, k % kPStages), ring_par(k));
}

// ---------------------------------------------------------------------------
// MMA issuers
// ---------------------------------------------------------------------------
// S_X = Q_X K^T for each tile that attends stage k, into S buffer k & 1, which
// is free once PV_X(k-2) has read the P written over it.  One thread issues
// every MMA of the CTA while two softmax warps share its SM sub-partition, so
// the descriptors of a stage are ready before its waits end: the issue itself
// is only the MMA instructions.
__device__ void pf_qk(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem)
{
    const uint32_t idesc = umma_idesc_bf16(128, kKT, false, false);
    // A (Q tile x) and B (K of a slot): one base descriptor each; the others
    // add (byte offset >> 4) to its 14-bit address field, which shared
    // addresses below 256 KB never carry out of
    uint64_t ad[kPTilesPerCta][kPHalves * 4];
#pragma unroll
    for (int x = 0; x < kPTilesPerCta; ++x)
#pragma unroll
        for (int i = 0; i < kPHalves * 4; ++i)
            ad[x][i] = umma_sdesc_sw128(c.base + c.lay.qtile + (uint32_t)(x * kPHalves * 128 * 128) +
                                            (uint32_t)((i >> 2) * 128 * 128 + (i & 3) * 32),
                                        16u, 1024u);
    const uint64_t kd0 = umma_sdesc_sw128(pf_slot(c, 0), 16u, 1024u);
    bool alive = pf_wait(pf_qready(c), 0u, c.abort_flag, p.err);
    for (int k = 0; k < t.nst_all; ++k) {
        const int slot = k % kPStages;
        uint64_t bd[kPHalves * 4];
#pragma unroll
        for (int i = 0; i < kPHalves * 4; ++i)
            bd[i] = kd0 + (((uint32_t)slot * c.lay.stage_bytes + (uint32_t)((i >> 2) * kKT * 128 + (i & 3) * 32)) >> 4);
        if (alive)
            alive = pf_wait(pf_full(c, false, slot), ring_par(k), c.abort_flag, p.err);
#pragma unroll
        for (int x = 0; x < kPTilesPerCta; ++x) {
            if (k >= t.nst[x])
                continue;
            if (alive && k >= 2)
                alive = pf_wait(pf_pvdone(c, x, k & 1), (uint32_t)(((k - 2) >> 1) & 1), c.abort_flag, p.err);
            if (alive) {
                tc_fence_after();
                const uint32_t d = tmem + col_s(x, k & 1);
#pragma unroll
                for (int i = 0; i < kPHalves * 4; ++i)
                    umma_bf16(d, ad[x][i], bd[i], idesc, i ? 1u : 0u);
            }
            umma_commit(pf_sfull(c, x, k & 1));
        }
        umma_commit(pf_empty(c, false, slot));
    }
    umma_commit(pf_fin(c));
    mbar_drain_bounded(pf_fin(c), 0u);
}

// O_X += P_X V; P_X from TMEM (over S buffer k & 1), V MN-major in the slot.  PV_A(k)
// waits for tile A's softmax, which also cleared the stage's unusable V rows
// for both tiles (tile B's alone once A no longer attends the stage).
__device__ void pf_pv(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem)
{
    const uint32_t idesc = umma_idesc_bf16(128, kPD, false, true);
    const uint64_t vd0 = umma_sdesc_sw128(pf_slot(c, 0) + (uint32_t)(kKT * kPD * 2), (uint32_t)(kKT * 128), 1024u);
    bool alive = true;
    for (int k = 0; k < t.nst_all; ++k) {
        const int slot = k % kPStages;
        uint64_t bd[kKT / 16];
#pragma unroll
        for (int ks = 0; ks < kKT / 16; ++ks)
            bd[ks] = vd0 + (((uint32_t)slot * c.lay.stage_bytes + (uint32_t)ks * 2048u) >> 4);
        if (alive)
            alive = pf_wait(pf_full(c, true, slot), ring_par(k), c.abort_flag, p.err);
#pragma unroll
        for (int x = 0; x < kPTilesPerCta; ++x) {
            if (k >= t.nst[x])
                continue;
            if (alive)
                alive = pf_wait(pf_pfull(c, x, k & 1), (uint32_t)((k >> 1) & 1), c.abort_flag, p.err);
            if (alive) {
                tc_fence_after();
                const uint32_t d = tmem + col_o(x);
                const uint32_t a = tmem + col_s(x, k & 1);
#pragma unroll
                for (int ks = 0; ks < kKT / 16; ++ks)
                    umma_bf16_ts(d, a + (uint32_t)(ks * 8), bd[ks], idesc, (k == 0 && ks == 0) ? 0u : 1u);
            }
            umma_commit(pf_pvdone(c, x, k & 1));
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
    const int P = p.page_size;
    const int log2P = 31 - __clz(P);
    const float sl2 = p.scale_log2;
    float m_use = -INFINITY, lsum = 0.f;
    bool alive = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        bool ok = false;
        if (alive)
            ok = pf_wait(bar, parity, c.abort_flag, p.err);
        alive = __all_sync(0xffffffffu, ok) && alive;
        return alive;
    };
    for (int k = 0; k < t.nst[x]; ++k) {
        const int slot = k % kPStages;
        const int key0 = k * kKT;
        const int buf = k & 1;
        const uint32_t srow = tmem + lane_base + col_s(x, buf);
        wait(pf_sfull(c, x, buf), (uint32_t)((k >> 1) & 1));
        wait(pf_full(c, true, slot), ring_par(k));           // V landed; orders the word below
        const uint32_t tagged = alive ? reinterpret_cast<const volatile uint32_t *>(c.smem + c.lay.meta)[slot] : 0u;
        if (alive && (tagged >> 8) != ((uint32_t)k & 0xffffffu)) {
            if (lane == 0) {
                atomicOr(p.err, SHKV_ERRF_PIPELINE);
                *c.abort_flag = 1u;
            }
            alive = false;
        }
        const uint32_t pmask = tagged & 0xffu;
        // keys this row may see: [key0, key0 + nvis), on pages that were copied
        const int nvis = row_ok ? min(kKT, pos - key0 + 1) : 0;
        const bool all_pages = pmask == (1u << (kKT / P)) - 1u;
        // no mask below the diagonal; padding rows (no token) need none either:
        // their scores only reach their own row of O, which is not stored
        const bool dense = alive && all_pages && (nvis == kKT || !row_ok);
        // 32 scores (already loaded), masked (-inf where invisible)
        auto mask_chunk = [&](int c32, uint32_t (&sv)[32]) {
            if (!dense) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int col = c32 * 32 + e;
                    const bool vis = alive && col < nvis && ((pmask >> (col >> log2P)) & 1u);
                    sv[e] = vis ? sv[e] : __float_as_uint(-INFINITY);
                }
            }
        };
        if (alive)
            tc_fence_after();
        // this row's 64 scores into registers
        uint32_t sv[2][32];
        tmem_ld32_nowait(srow, sv[0]);
        tmem_ld32_nowait(srow + 32u, sv[1]);
        tmem_wait_ld();
        mask_chunk(0, sv[0]);
        mask_chunk(1, sv[1]);
        float cm;
        {
            float a = -INFINITY, b = -INFINITY, d = -INFINITY, e4 = -INFINITY;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    a = max3f(a, __uint_as_float(sv[h][e]), __uint_as_float(sv[h][e + 1]));
                    b = max3f(b, __uint_as_float(sv[h][e + 2]), __uint_as_float(sv[h][e + 3]));
                    d = max3f(d, __uint_as_float(sv[h][e + 4]), __uint_as_float(sv[h][e + 5]));
                    e4 = max3f(e4, __uint_as_float(sv[h][e + 6]), __uint_as_float(sv[h][e + 7]));
                }
            cm = max3f(a, b, fmaxf(d, e4));
        }
        // the running maximum moves only by more than 2^kPRescaleLog2 (or
        // when it is first set; O and the sum are still zero then)
        const float mt = cm * sl2;                                // sl2 > 0; -inf if nothing is visible
        const bool first = m_use == -INFINITY && mt != -INFINITY;
        const bool need = alive && m_use != -INFINITY && mt > m_use + kPRescaleLog2;
        if (first)
            m_use = mt;
        if (__any_sync(0xffffffffu, need)) {
            // tcgen05.ld/st are warp-wide: lanes that keep their maximum scale by 1
            const float alpha = need ? ex2_approx(m_use - mt) : 1.f;
            if (k >= 1) {
                wait(pf_pvdone(c, x, (k - 1) & 1), (uint32_t)(((k - 1) >> 1) & 1));
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
        // P = 2^(s * scale_log2 - m) as bf16 pairs over columns 0 .. 31 of
        // the S buffer (the scores are in registers)
        const float mu = m_use == -INFINITY ? 0.f : m_use;
        float part = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float pp[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float p0 = ex2_approx(fmaf(__uint_as_float(sv[h][2 * e]), sl2, -mu));
                const float p1 = ex2_approx(fmaf(__uint_as_float(sv[h][2 * e + 1]), sl2, -mu));
                pp[e & 3] += p0 + p1;
                pk[e] = pack_bf16x2(p0, p1);
            }
            tmem_st16_nowait(srow + (uint32_t)(h * 16), pk);
            part += (pp[0] + pp[1]) + (pp[2] + pp[3]);
        }
        lsum += part;
        tmem_wait_st();
        tc_fence_before();
        // V rows of keys that no row may use in this stage (past the request's
        // end, or on a skipped page) may hold stale or non-finite bits: zero
        // them (thread r takes key row r).  Tile A does it while it attends the
        // stage, tile B after that.
        if (x == 0 || k >= t.nst[0]) {
            const int key = key0 + r;
            const bool zero_mine = alive && r < kKT && !(key < t.L && ((pmask >> (r >> log2P)) & 1u));
            if (__any_sync(0xffffffffu, zero_mine)) {
                if (zero_mine) {
                    const uint32_t vrow = pf_slot(c, slot) + (uint32_t)(kKT * kPD * 2) + (uint32_t)r * 128u;
#pragma unroll
                    for (int h = 0; h < kPHalves; ++h)
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch)
                            st_shared_zero16(vrow + (uint32_t)(h * kKT * 128 + ch * 16));
                }
                fence_proxy_async_smem();
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(pf_pfull(c, x, buf));
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
    bool ok = alive && pf_wait(pf_pvdone(c, x, last & 1), (uint32_t)((last >> 1) & 1), c.abort_flag, p.err);
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
        for (int s = 0; s < kPStages; ++s)
            for (int v = 0; v < 2; ++v) {
                mbar_init(pf_full(c, v, s), 1);
                mbar_init(pf_empty(c, v, s), 1);
            }
        for (int x = 0; x < kPTilesPerCta; ++x) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(pf_sfull(c, x, b), 1);
                mbar_init(pf_pfull(c, x, b), kPGroupWarps);
                mbar_init(pf_pvdone(c, x, b), 1);
            }
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
    } else {
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
            const uint32_t qtile = c.lay.qtile + (uint32_t)(x * kPHalves * 128 * 128);
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
    cudaError_t e = cudaFuncSetAttribute(shkv_prefill_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess)
        return e;
    shkv_prefill_umma_kernel<<<grid, kPThreads, smem, stream>>>(tmK, tmV, p);
    return cudaGetLastError();
}

}  // namespace shkv
