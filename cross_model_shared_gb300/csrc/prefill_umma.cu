// prefill_umma.cu -- causal partial-prefill attention on the 5th-generation
// tensor cores (tcgen05 / TMEM), head dim 128.
//
// PrefillShare Sec. 3.3: on a prefix-cache hit the shared prefill module runs
// only on the n_new new tokens and extends the cached prefix.  Their K/V have
// been appended to the paged pool, so request b holds L_b tokens, the last
// n_new of them new; new token i sits at position L_b - n_new + i and
// attends every key at a position <= its own.
//
// One CTA per (request, KV head, tile of new tokens).  The tile's 128 MMA rows
// are TPT = floor(128 / G) new tokens x the G query heads of the KV head
// (row r = i * G + j), so every K/V page is read once for the whole group.
// Per 128-key stage:
//   S[r, key]  = sum_d Q[r, d] K[key, d]      M = 128 rows, N = 128 keys
//   O[r, d]   += sum_key P[r, key] V[key, d]  M = 128 rows, N = 128 = D
// S (two buffers) and O live in TMEM; a softmax thread owns one row (its TMEM
// lane), keeps its running max and sum, and rescales its own row of O lazily
// (only when the max rises by more than 2^kRescaleLog2).  P (bf16) is written
// over the stage's K tile, which the QK MMA has consumed.  Key stages past
// the tile's last position are never loaded; on the diagonal the causal mask
// is applied per element.
//
// Roles (224 threads): warps 0-3 softmax (row = TMEM lane), warp 4 QK issuer,
// warp 5 PV issuer (its commit frees the ring slot), warp 6 producer (TMA of
// K and V page halves, one box per lane).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "shkv_device.cuh"

namespace shkv {


namespace {

constexpr int kKT = 128;                 // keys per stage
constexpr int kPD = 128;                 // head dim
constexpr int kPHalves = kPD / 64;
constexpr int kPThreads = 224;
constexpr int kPSoftmaxWarps = 4;
constexpr int kPQkWarp = 4;
constexpr int kPPvWarp = 5;
constexpr int kPProducerWarp = 6;
constexpr uint32_t kPTmemCols = 512;
constexpr uint32_t kPColS = 0;           // S buffers at 0 and 128
constexpr uint32_t kPColO = 256;
constexpr float kPRescaleLog2 = 8.f;
constexpr int kPMaxStages = 3;

struct PfSmem {
    uint32_t ring, stage_bytes, qtile, bars, meta, misc, tslot, total;
};

// ring slots of [K | V][half][128 keys][128 B], then the Q tile
// [half][128 rows][128 B] (both 128-byte swizzled), then the barriers:
// full[S], empty[S], p_full[S], s_full[2], s_free[2], fin
__host__ __device__ inline PfSmem pf_layout(int stages)
{
    PfSmem u;
    u.stage_bytes = (uint32_t)(2 * kKT * kPD * 2);
    u.ring = 0;
    u.qtile = (uint32_t)stages * u.stage_bytes;
    u.bars = u.qtile + (uint32_t)(kPHalves * 128 * 128);
    u.meta = u.bars + (uint32_t)((3 * stages + 5) * 8);
    u.misc = u.meta + (uint32_t)(stages * 4);
    u.tslot = u.misc + 8;
    u.total = u.misc + 16 + 1024;
    return u;
}

struct PfCtx {
    uint8_t *smem;
    uint32_t base;
    PfSmem lay;
    int stages;
    volatile uint32_t *abort_flag;
};

__device__ __forceinline__ uint32_t pbar(const PfCtx &c, int i) { return c.base + c.lay.bars + 8u * i; }
__device__ __forceinline__ uint32_t pf_full(const PfCtx &c, int s) { return pbar(c, s); }
__device__ __forceinline__ uint32_t pf_empty(const PfCtx &c, int s) { return pbar(c, c.stages + s); }
__device__ __forceinline__ uint32_t pf_pfull(const PfCtx &c, int s) { return pbar(c, 2 * c.stages + s); }
__device__ __forceinline__ uint32_t pf_sfull(const PfCtx &c, int b) { return pbar(c, 3 * c.stages + b); }
__device__ __forceinline__ uint32_t pf_sfree(const PfCtx &c, int b) { return pbar(c, 3 * c.stages + 2 + b); }
__device__ __forceinline__ uint32_t pf_fin(const PfCtx &c) { return pbar(c, 3 * c.stages + 4); }
__device__ __forceinline__ uint32_t pf_slot(const PfCtx &c, int s)
{
    return c.base + c.lay.ring + (uint32_t)s * c.lay.stage_bytes;
}

// the tile this CTA owns
struct Tile {
    int b, g, i0, ntok;          // request, KV head, first new token, new tokens in the tile
    int L, prefix;               // request length (with the new tokens), cached tokens before them
    int nst;                     // key stages: keys 0 .. last position
};

__device__ __forceinline__ Tile pf_tile(const PrefillParams &p)
{
    Tile t;
    int idx = blockIdx.x;
    const int qt = idx % p.tiles;
    idx /= p.tiles;
    t.g = idx % p.hkv;
    t.b = idx / p.hkv;
    t.i0 = qt * p.tpt;
    t.ntok = min(p.tpt, p.n_new - t.i0);
    t.L = p.lens[t.b];
    t.prefix = t.L - p.n_new;
    const int last_pos = t.prefix + t.i0 + t.ntok - 1;
    t.nst = last_pos / kKT + 1;
    return t;
}

// ---------------------------------------------------------------------------
// producer: stage k = keys [128k, 128k + 128), 128/P pages, K and V halves
// ---------------------------------------------------------------------------
__device__ void pf_producer(const CUtensorMap *tmK, const CUtensorMap *tmV, const PrefillParams &p,
                            const PfCtx &c, const Tile &t)
{
    const int lane = threadIdx.x & 31;
    const int P = p.page_size;
    const int RB = kKT / P;
    const int per_tensor = kPHalves * RB;
    const bool my_v = lane >= per_tensor;
    const int cl = my_v ? lane - per_tensor : lane;
    const int my_h = cl / RB, my_rb = cl % RB;
    const bool copier = lane < 2 * per_tensor;
    const uint32_t page_bytes = kPHalves * (uint32_t)P * 128u;
    const uint64_t pol = l2_evict_first_policy();
    if (lane == 0) {
        prefetch_tensormap(tmK);
        prefetch_tensormap(tmV);
        if (__ldg(p.seq_lens + t.b) != t.L)
            atomicOr(p.err, SHKV_ERRF_SEQ_LEN);
    }
    const int npages = (t.L + P - 1) / P;
    const int32_t *btrow = p.block_table + (int64_t)t.b * p.max_pages;
    bool alive = true;
    int last_issued = -1;
    for (int k = 0; k < t.nst; ++k) {
        const int slot = k % c.stages;
        const int pg = (k * kKT) / P + my_rb;
        const int my_id = (copier && pg < npages) ? __ldg(btrow + pg) : -1;
        bool ok = true;
        if (alive && lane == 0)
            ok = mbar_wait_bounded(pf_empty(c, slot), (uint32_t)(((k / c.stages) & 1) ^ 1), c.abort_flag, p.err);
        alive = alive && __all_sync(0xffffffffu, ok);
        const bool my_valid = copier && pg < npages && my_id >= 0 && my_id < p.num_pages;
        const uint32_t mask = __ballot_sync(0xffffffffu, my_valid) & ((1u << RB) - 1u);
        if (alive && lane == 0) {
            for (int rb = 0; rb < RB; ++rb)
                if (!((mask >> rb) & 1u) && (k * kKT) / P + rb < npages)
                    atomicOr(p.err, SHKV_ERRF_PAGE_OOB);
            reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.meta)[slot] = mask | ((uint32_t)k << 8);
            mbar_arrive_expect_tx(pf_full(c, slot), (uint32_t)__popc(mask) * page_bytes * 2u);
        }
        __syncwarp();
        if (alive && my_valid) {
            const uint32_t dst = pf_slot(c, slot) + (my_v ? (uint32_t)(kKT * kPD * 2) : 0u) +
                                 (uint32_t)my_h * (kKT * 128) + (uint32_t)my_rb * (uint32_t)P * 128u;
            tma_load_2d(dst, my_v ? tmV : tmK, my_h * 64, (my_id * p.hkv + t.g) * P, pf_full(c, slot), pol);
        }
        if (alive)
            last_issued = k;
        __syncwarp();
    }
    if (!alive && lane == 0)
        for (int k = last_issued - c.stages + 1; k <= last_issued; ++k)
            if (k >= 0)
                mbar_drain_bounded(pf_full(c, k % c.stages), (uint32_t)((k / c.stages) & 1));
}

// ---------------------------------------------------------------------------
// MMA issuers
// ---------------------------------------------------------------------------
__device__ void pf_qk(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem)
{
    const uint32_t idesc = umma_idesc_bf16(128, kKT, false, false);
    const uint32_t qtile = c.base + c.lay.qtile;
    bool alive = true;
    for (int k = 0; k < t.nst; ++k) {
        const int slot = k % c.stages, buf = k & 1;
        if (alive)
            alive = mbar_wait_bounded(pf_full(c, slot), (uint32_t)((k / c.stages) & 1), c.abort_flag, p.err);
        if (alive)
            alive = mbar_wait_bounded(pf_sfree(c, buf), (uint32_t)(((k >> 1) & 1) ^ 1), c.abort_flag, p.err);
        if (alive) {
            tc_fence_after();
            const uint32_t kst = pf_slot(c, slot);
#pragma unroll
            for (int h = 0; h < kPHalves; ++h)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = umma_sdesc_sw128(qtile + (uint32_t)(h * 128 * 128 + kk * 32), 16u, 1024u);
                    const uint64_t bd = umma_sdesc_sw128(kst + (uint32_t)(h * kKT * 128 + kk * 32), 16u, 1024u);
                    umma_bf16(tmem + kPColS + (uint32_t)(buf * kKT), ad, bd, idesc, (h | kk) ? 1u : 0u);
                }
        }
        umma_commit(pf_sfull(c, buf));
    }
    umma_commit(pf_fin(c));
    mbar_drain_bounded(pf_fin(c), 0u);
}

// O += P V; P over the slot's K region ([key half][row][128 B]), V MN-major
__device__ void pf_pv(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem)
{
    const uint32_t idesc = umma_idesc_bf16(128, kPD, false, true);
    bool alive = true;
    for (int k = 0; k < t.nst; ++k) {
        const int slot = k % c.stages;
        if (alive)
            alive = mbar_wait_bounded(pf_pfull(c, slot), (uint32_t)((k / c.stages) & 1), c.abort_flag, p.err);
        if (alive) {
            tc_fence_after();
            const uint32_t kst = pf_slot(c, slot);
            const uint32_t vst = kst + (uint32_t)(kKT * kPD * 2);
#pragma unroll
            for (int ks = 0; ks < kKT / 16; ++ks) {
                const uint64_t ad =
                    umma_sdesc_sw128(kst + (uint32_t)((ks >> 2) * (128 * 128) + (ks & 3) * 32), 16u, 1024u);
                const uint64_t bd = umma_sdesc_sw128(vst + (uint32_t)ks * 2048u, (uint32_t)(kKT * 128), 1024u);
                umma_bf16(tmem + kPColO, ad, bd, idesc, (k == 0 && ks == 0) ? 0u : 1u);
            }
        }
        umma_commit(pf_empty(c, slot));
    }
    umma_commit(pf_fin(c));
    mbar_drain_bounded(pf_fin(c), 0u);
}

// ---------------------------------------------------------------------------
// softmax warps: thread r = MMA row r = (new token i0 + r / G, head r % G)
// ---------------------------------------------------------------------------
__device__ void pf_softmax(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem, float &m_out,
                           float &l_out, bool &alive_out)
{
    const int r = threadIdx.x;
    const int lane = r & 31, warp = r >> 5;
    const int ti = r / p.group, tj = r - (r / p.group) * p.group;
    const bool row_ok = ti < t.ntok;
    const int pos = t.prefix + t.i0 + ti;                // this row's position (keys 0 .. pos)
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int P = p.page_size;
    const int log2P = 31 - __clz(P);
    const float sl2 = p.scale_log2;
    float m_use = -INFINITY, lsum = 0.f;
    bool alive = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        bool ok = false;
        if (alive)
            ok = mbar_wait_bounded(bar, parity, c.abort_flag, p.err);
        alive = __all_sync(0xffffffffu, ok) && alive;
        return alive;
    };
    for (int k = 0; k < t.nst; ++k) {
        const int slot = k % c.stages, buf = k & 1;
        const int key0 = k * kKT;
        wait(pf_sfull(c, buf), (uint32_t)((k >> 1) & 1));
        wait(pf_full(c, slot), (uint32_t)((k / c.stages) & 1));      // (complete already: orders the word below)
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
        const bool dense = alive && nvis == kKT && all_pages;    // below the diagonal: no mask
        const uint32_t srow = tmem + lane_base + kPColS + (uint32_t)(buf * kKT);
        uint8_t *prow = c.smem + c.lay.ring + (uint32_t)slot * c.lay.stage_bytes + (uint32_t)r * 128u;
        // 32 scores of this row from TMEM, masked (-inf where invisible)
        auto load_chunk = [&](int c32, uint32_t (&sv)[32]) {
            tmem_ld32(srow + (uint32_t)(c32 * 32), sv);
            if (!dense) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int col = c32 * 32 + e;
                    const bool vis = alive && col < nvis && ((pmask >> (col >> log2P)) & 1u);
                    sv[e] = vis ? sv[e] : __float_as_uint(-INFINITY);
                }
            }
        };
        // P of 32 keys (bf16) over the consumed K tile: keys 0..63 in half 0, 64..127 in half 1
        auto emit_chunk = [&](int c32, const uint32_t (&sv)[32], float mu, bool store) -> float {
            float part = 0.f;
#pragma unroll
            for (int q8 = 0; q8 < 4; ++q8) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = q8 * 8 + 2 * e;
                    const float p0 = ex2_approx(fmaf(__uint_as_float(sv[i]), sl2, -mu));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(sv[i + 1]), sl2, -mu));
                    part += p0 + p1;
                    pk[e] = pack_bf16x2(p0, p1);
                }
                const int ch = c32 * 4 + q8;                      // 16-byte chunk of the 256-byte row
                if (store)
                    *reinterpret_cast<uint4 *>(prow + (uint32_t)(ch >> 3) * (128u * 128u) +
                                               (((ch & 7) ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            return part;
        };
        if (alive)
            tc_fence_after();
        // a row with no running max yet takes this stage's max first
        if (__any_sync(0xffffffffu, alive && m_use == -INFINITY && nvis > 0)) {
            float cm = -INFINITY;
#pragma unroll 1
            for (int c32 = 0; c32 < kKT / 32; ++c32) {
                uint32_t sv[32];
                load_chunk(c32, sv);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    cm = fmaxf(cm, __uint_as_float(sv[e]));
            }
            if (m_use == -INFINITY)
                m_use = cm * sl2;                                 // sl2 > 0; stays -inf if nothing is visible
        }
        // stream the row: exponents against the running max, tracking this stage's max
        const float l_before = lsum;
        const float mu = m_use == -INFINITY ? 0.f : m_use;
        float cmax = -INFINITY, part = 0.f;
#pragma unroll 1
        for (int c32 = 0; c32 < kKT / 32; ++c32) {
            uint32_t sv[32];
            load_chunk(c32, sv);
#pragma unroll
            for (int e = 0; e < 32; ++e)
                cmax = fmaxf(cmax, __uint_as_float(sv[e]));
            part += emit_chunk(c32, sv, mu, alive);
        }
        lsum += part;
        // lazy refresh: a row whose max rose by more than 2^kPRescaleLog2
        // rescales its O (after the previous PV) and redoes this stage's P
        // from S, still in TMEM.  tcgen05.ld/st are warp-wide, so the whole
        // warp takes part (scale 1, no rewrite, where nothing moved).
        const float mt = cmax * sl2;
        const bool need = alive && m_use != -INFINITY && mt > m_use + kPRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
            const float alpha = need ? ex2_approx(m_use - mt) : 1.f;
            if (k >= 1) {
                const int kp = k - 1;
                wait(pf_empty(c, kp % c.stages), (uint32_t)((kp / c.stages) & 1));
                if (alive) {
                    tc_fence_after();
#pragma unroll 1
                    for (int c32 = 0; c32 < kPD / 32; ++c32) {
                        uint32_t ov[32];
                        tmem_ld32(tmem + lane_base + kPColO + (uint32_t)(c32 * 32), ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st32(tmem + lane_base + kPColO + (uint32_t)(c32 * 32), ov);
                    }
                }
            }
            if (need)
                m_use = mt;
            float redo = 0.f;
#pragma unroll 1
            for (int c32 = 0; c32 < kKT / 32; ++c32) {
                uint32_t sv[32];
                if (alive)
                    load_chunk(c32, sv);
                redo += emit_chunk(c32, sv, m_use, alive && need);
            }
            if (need)
                lsum = l_before * alpha + redo;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(pf_sfree(c, buf));
        // V rows of keys that no row may use in this stage (past the request's
        // end, or on a skipped page) may hold stale or non-finite bits: zero
        // them (thread r takes key row r)
        {
            const int key = key0 + r;
            const bool key_ok = key < t.L && ((pmask >> (r >> log2P)) & 1u);
            if (alive && !key_ok) {
                const uint32_t vrow = pf_slot(c, slot) + (uint32_t)(kKT * kPD * 2) + (uint32_t)r * 128u;
#pragma unroll
                for (int h = 0; h < kPHalves; ++h)
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_zero16(vrow + (uint32_t)(h * kKT * 128 + ch * 16));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0)
            mbar_arrive(pf_pfull(c, slot));
    }
    m_out = m_use;
    l_out = lsum;
    alive_out = alive;
}

// ---------------------------------------------------------------------------
// epilogue: this row of O, normalised, and its log-sum-exp
// ---------------------------------------------------------------------------
__device__ void pf_epilogue(const PrefillParams &p, const PfCtx &c, const Tile &t, uint32_t tmem, float m_use,
                            float lsum, bool alive)
{
    const int r = threadIdx.x;
    const int warp = r >> 5;
    const int ti = r / p.group, tj = r - (r / p.group) * p.group;
    const bool row_ok = ti < t.ntok;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const int last = t.nst - 1;
    bool ok = alive && mbar_wait_bounded(pf_empty(c, last % c.stages), (uint32_t)((last / c.stages) & 1),
                                         c.abort_flag, p.err);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok)
        return;
    tc_fence_after();
    const float inv = lsum > 0.f ? __frcp_rn(lsum) : 0.f;
    const int64_t row = ((int64_t)t.b * p.n_new + t.i0 + ti) * p.hq + (int64_t)t.g * p.group + tj;
#pragma unroll 1
    for (int c32 = 0; c32 < kPD / 32; ++c32) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + kPColO + (uint32_t)(c32 * 32), ov);
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
    c.stages = p.stages;
    c.lay = pf_layout(p.stages);
    c.abort_flag = reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.misc);
    const Tile t = pf_tile(p);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < c.stages; ++s) {
            mbar_init(pf_full(c, s), 1);
            mbar_init(pf_empty(c, s), 1);
            mbar_init(pf_pfull(c, s), kPSoftmaxWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(pf_sfull(c, i), 1);
            mbar_init(pf_sfree(c, i), kPSoftmaxWarps);
        }
        mbar_init(pf_fin(c), 2);
        *c.abort_flag = 0u;
        fence_barrier_init();
    }
    if (warp < kPSoftmaxWarps) {
        // this thread's query row into the swizzled K-major Q tile (padding rows zero)
        const int r = threadIdx.x;
        const int ti = r / p.group, tj = r - (r / p.group) * p.group;
        const bool row_ok = ti < t.ntok;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            p.q + (((int64_t)t.b * p.n_new + t.i0 + ti) * p.hq + (int64_t)t.g * p.group + tj) * kPD);
#pragma unroll
        for (int ch = 0; ch < kPD / 8; ++ch) {
            const uint4 v = row_ok ? __ldg(src + ch) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t off = (uint32_t)(ch >> 3) * (128u * 128u) + (uint32_t)r * 128u +
                                 (uint32_t)(((ch & 7) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4 *>(c.smem + c.lay.qtile + off) = v;
        }
        fence_proxy_async_smem();
    }
    if (warp == 0)
        tmem_alloc(c.base + c.lay.tslot, kPTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.tslot);

    if (warp == kPProducerWarp)
        pf_producer(&tmK, &tmV, p, c, t);
    else if (warp == kPQkWarp) {
        if ((threadIdx.x & 31) == 0)
            pf_qk(p, c, t, tmem);
    } else if (warp == kPPvWarp) {
        if ((threadIdx.x & 31) == 0)
            pf_pv(p, c, t, tmem);
    } else if (warp < kPSoftmaxWarps) {
        float m_use, lsum;
        bool alive;
        pf_softmax(p, c, t, tmem, m_use, lsum, alive);
        pf_epilogue(p, c, t, tmem, m_use, lsum, alive);
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
int prefill_stages()
{
    int st = kPMaxStages;
    while (st >= 2 && pf_layout(st).total > (uint32_t)kSmemLimit)
        --st;
    return st;
}

uint32_t prefill_smem_bytes(int stages) { return pf_layout(stages).total; }

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
