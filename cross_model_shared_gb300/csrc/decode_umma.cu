// decode_umma.cu -- shared-KV decode attention on the 5th-generation tensor
// cores (tcgen05 / TMEM), for many stacked rows per KV head.
//
// Same method and work split as decode_attn.cu (ICaRus key design 3 over the
// PrefillShare paged cache; persistent CTAs over cost-balanced chunk
// ranges; split units merged by the last arriving CTA), with the consumer
// side rebuilt around tcgen05.mma:
//
//   warp 3  producer: TMA of K/V row-blocks into the mbarrier ring and bulk
//           copies of each segment's query rows (shared with decode_attn.cu);
//   warp 2  MMA issuer (one lane): S = Q K^T into a double-buffered TMEM
//           tile (M = 128 query-row lanes, N = the stage's tokens), one stage
//           ahead of O += P V (V read MN-major straight from the ring slot);
//   warps 0-1 softmax: one thread per stacked row (TMEM lanes 0..63).  Each
//           reads its row of S from TMEM, masks, keeps a base-2 running max
//           and sum, writes its row of P (bf16) to a swizzled shared tile, and
//           at the end of a segment reads its row of O from TMEM.  The running
//           max is refreshed lazily: O (in TMEM) is rescaled only when a tile
//           raises a row's max by more than 2^8, so P stays below 256.
//
// Because every row lives in exactly one thread, there is no cross-warp
// combine at a segment end.  Rows R..127 of the MMA tiles are padding: they
// read whatever the shared memory holds and their results are never used.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "decode_common.cuh"

namespace shkv {

namespace {

using namespace detail;

static_assert(kStageTokens == 32, "the tcgen05 consumer reads 32 tokens of S per stage");

constexpr int kUmmaThreads = 128;
constexpr int kSoftmaxWarps = 2;            // TMEM lanes 0..63: up to 64 stacked rows
constexpr int kMmaWarp = 2;
constexpr int kProducerWarp = 3;
constexpr uint32_t kTmemCols = 256;         // S[2] (2 x 32 columns) + O (up to 128 columns)
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 64;
constexpr float kRescaleLog2 = 8.f;
constexpr float kLn2u = 0.6931471805599453f;

// extra barriers: s_full[2], s_free[2], p_full[2], p_free[2], q_ready, q_tile_free, fin
constexpr int kNumXbars = 11;

struct UmmaSmem {
    DecodeSmem s;     // ring, Q staging, ring/Q barriers, meta, misc (shared with the producer)
    uint32_t qtile;   // Q as the A operand: [D/64 halves][128 rows][128 B], swizzled
    uint32_t ptile0;  // P tiles ([rows][128 B], swizzled) in the unused rows 64..127 of the Q tile
    uint32_t ptile1;
    uint32_t xbars;
    uint32_t tslot;   // TMEM base address written by tcgen05.alloc
};

__host__ __device__ inline UmmaSmem umma_smem_layout(int D, int rows, int stages)
{
    UmmaSmem u;
    DecodeSmem &s = u.s;
    const uint32_t half_bytes = 128u * 128u;        // one column half of the 128-row Q tile
    s.stage_bytes = (uint32_t)(2 * kStageTokens * D * 2);
    s.ring = 0;
    u.qtile = s.ring + (uint32_t)stages * s.stage_bytes;
    u.ptile0 = u.qtile + 64u * 128u;                // half 0, rows 64..127
    u.ptile1 = D >= 128 ? u.qtile + half_bytes + 64u * 128u : u.qtile + half_bytes;
    const uint32_t qtile_end = u.qtile + (uint32_t)(D / 64) * half_bytes + (D >= 128 ? 0u : 64u * 128u);
    s.qbuf = align_up(qtile_end > u.ptile1 + 64u * 128u ? qtile_end : u.ptile1 + 64u * 128u, 128);
    s.qbuf_bytes = align_up((uint32_t)(rows * D * 2), 128);
    s.comb_o = s.comb_m = s.comb_l = 0;
    s.bars = align_up(s.qbuf + 2 * s.qbuf_bytes, 8);
    u.xbars = s.bars + (uint32_t)((2 * stages + 4) * 8);
    s.meta = u.xbars + (uint32_t)(kNumXbars * 8);
    s.misc = s.meta + (uint32_t)(stages * 4);
    u.tslot = s.misc + 8;
    // The MMAs read both P tiles and the Q tile as full 128-row operands, so
    // the padding rows of the last tile must also lie inside the allocation.
    const uint32_t mma_end = u.ptile1 + 128u * 128u;
    const uint32_t used = s.misc + 16 > mma_end ? s.misc + 16 : mma_end;
    s.total = used + 1024;   // + slack to align the base to 1024 bytes
    return u;
}

struct UCtx {
    Ctx c;
    UmmaSmem u;
};

__device__ __forceinline__ uint32_t xbar(const UCtx &x, int i) { return x.c.base + x.u.xbars + 8u * i; }
__device__ __forceinline__ uint32_t s_full_bar(const UCtx &x, int b) { return xbar(x, 0 + b); }
__device__ __forceinline__ uint32_t s_free_bar(const UCtx &x, int b) { return xbar(x, 2 + b); }
__device__ __forceinline__ uint32_t p_full_bar(const UCtx &x, int b) { return xbar(x, 4 + b); }
__device__ __forceinline__ uint32_t p_free_bar(const UCtx &x, int b) { return xbar(x, 6 + b); }
__device__ __forceinline__ uint32_t q_ready_bar(const UCtx &x) { return xbar(x, 8); }
__device__ __forceinline__ uint32_t q_tile_free_bar(const UCtx &x) { return xbar(x, 9); }
__device__ __forceinline__ uint32_t fin_bar(const UCtx &x) { return xbar(x, 10); }

__device__ __forceinline__ uint32_t ptile(const UCtx &x, int b) { return x.c.base + (b ? x.u.ptile1 : x.u.ptile0); }

// ---------------------------------------------------------------------------
// MMA issuer (one lane)
// ---------------------------------------------------------------------------
template <int D>
__device__ void mma_issuer(const DecodeParams &p, const UCtx &x, uint32_t tmem)
{
    constexpr int TT = kStageTokens;
    constexpr int HALVES = D / 64;
    const Ctx &c = x.c;
    const int stages = p.stages;
    const int P = p.page_size;
    const int BR = p.box_rows;
    const int RB = TT / BR;
    const uint32_t idesc_qk = umma_idesc_bf16(128, BR, false, false);
    const uint32_t idesc_pv = umma_idesc_bf16(128, D, false, true);
    const uint32_t qtile = c.base + x.u.qtile;
    bool alive = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (alive)
            alive = mbar_wait_bounded(bar, parity, c.abort_flag, p.err);
        return alive;
    };

    // O += P(k) V(k) for stage k of the current segment
    auto pv = [&](int k, bool first) {
        const int buf = k & 1;
        const int slot = k % stages;
        if (wait(p_full_bar(x, buf), (uint32_t)((k >> 1) & 1))) {
            tc_fence_after();
            const uint32_t vst = c.base + c.lay.ring + (uint32_t)slot * c.lay.stage_bytes + (uint32_t)(TT * D * 2);
#pragma unroll
            for (int ks = 0; ks < TT / 16; ++ks) {
                const int t0 = ks * 16;
                const uint32_t va = vst + (uint32_t)((t0 / BR) * (BR * D * 2) + (t0 % BR) * 128);
                const uint64_t bd = umma_sdesc_sw128(va, (uint32_t)(BR * 128), 1024u);
                const uint64_t ad = umma_sdesc_sw128(ptile(x, buf) + (uint32_t)(ks * 32), 16u, 1024u);
                umma_bf16(tmem + kTmemO, ad, bd, idesc_pv, (first && ks == 0) ? 0u : 1u);
            }
        }
        umma_commit(empty_bar(c, slot, stages));
        umma_commit(p_free_bar(x, buf));
    };

    int kbase = 0, seg = 0;
    Segment s = locate(p, c.cta_begin, c.cta_end);
    for (;;) {
        const int nst = (s.p1 * P - s.p0 * P + TT - 1) / TT;
        wait(q_ready_bar(x), (uint32_t)(seg & 1));
        tc_fence_after();
        for (int j = 0; j < nst; ++j) {
            const int k = kbase + j;
            const int buf = k & 1;
            const int slot = k % stages;
            wait(full_bar(c, slot), (uint32_t)((k / stages) & 1));
            wait(s_free_bar(x, buf), (uint32_t)(((k >> 1) & 1) ^ 1));
            if (alive) {
                tc_fence_after();
                const uint32_t kst = c.base + c.lay.ring + (uint32_t)slot * c.lay.stage_bytes;
                for (int rb = 0; rb < RB; ++rb) {
#pragma unroll
                    for (int h = 0; h < HALVES; ++h)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = umma_sdesc_sw128(qtile + (uint32_t)(h * 128 * 128 + kk * 32), 16u, 1024u);
                            const uint64_t bd = umma_sdesc_sw128(
                                kst + (uint32_t)(rb * (BR * D * 2) + h * (BR * 128) + kk * 32), 16u, 1024u);
                            umma_bf16(tmem + kTmemS + (uint32_t)(buf * TT + rb * BR), ad, bd, idesc_qk,
                                      (h | kk) ? 1u : 0u);
                        }
                }
            }
            umma_commit(s_full_bar(x, buf));
            if (j >= 1)
                pv(k - 1, j == 1);
        }
        pv(kbase + nst - 1, nst == 1);
        umma_commit(q_tile_free_bar(x));
        kbase += nst;
        ++seg;
        if (s.seg_end >= c.cta_end)
            break;
        s = next_segment(p, s, c.cta_end);
    }
    // every MMA issued above has completed once this arrives
    umma_commit(fin_bar(x));
    mbar_drain_bounded(fin_bar(x), 0u);
}

// ---------------------------------------------------------------------------
// softmax warps (thread = stacked row)
// ---------------------------------------------------------------------------
template <int D>
__device__ void softmax_rows(const DecodeParams &p, const UCtx &x, uint32_t tmem)
{
    constexpr int TT = kStageTokens;
    const Ctx &c = x.c;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r = warp * 32 + lane;            // stacked row == TMEM lane
    const bool active = r < p.rows;
    const int stages = p.stages;
    const int P = p.page_size;
    const int BR = p.box_rows;
    const int log2BR = 31 - __clz(BR);
    const float sl2 = p.scale_log2;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const volatile uint32_t *meta = reinterpret_cast<const volatile uint32_t *>(c.smem + c.lay.meta);
    bool alive = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
        bool ok = false;
        if (alive)
            ok = mbar_wait_bounded(bar, parity, c.abort_flag, p.err);
        alive = __all_sync(0xffffffffu, ok) && alive;
        return alive;
    };

    int kbase = 0, seg = 0;
    Segment s = locate(p, c.cta_begin, c.cta_end);
    for (;;) {
        const int tok_end = s.p1 * P;
        const int nst = (tok_end - s.p0 * P + TT - 1) / TT;
        const int L = plan_len(p, s);
        const int lim = L < tok_end ? L : tok_end;

        // --- query row r: staging buffer -> swizzled Q tile (A operand)
        if (seg > 0)
            wait(q_tile_free_bar(x), (uint32_t)((seg - 1) & 1));
        const int qb = seg & 1;
        wait(qfull_bar(c, qb, stages), (uint32_t)((seg >> 1) & 1));
        if (alive && active) {
            const uint8_t *src = c.smem + c.lay.qbuf + qb * c.lay.qbuf_bytes + (size_t)r * D * 2;
#pragma unroll
            for (int ch = 0; ch < D / 8; ++ch) {
                const uint4 v = *reinterpret_cast<const uint4 *>(src + ch * 16);
                const uint32_t off = (uint32_t)((ch >> 3) * 128 * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
                *reinterpret_cast<uint4 *>(c.smem + x.u.qtile + off) = v;
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(qempty_bar(c, qb, stages));
            mbar_arrive(q_ready_bar(x));
        }

        float m_use = -INFINITY, lsum = 0.f;
        for (int j = 0; j < nst; ++j) {
            const int k = kbase + j;
            const int buf = k & 1;
            const int slot = k % stages;
            // --- this row of S for the stage's tokens
            uint32_t sv[32];
            if (wait(s_full_bar(x, buf), (uint32_t)((k >> 1) & 1))) {
                tc_fence_after();
                tmem_ld32(tmem + lane_base + kTmemS + (uint32_t)(buf * TT), sv);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(s_free_bar(x, buf));
            // the slot's TMA data (V rows to mask, the validity word)
            wait(full_bar(c, slot), (uint32_t)((k / stages) & 1));
            const uint32_t tagged = alive ? meta[slot] : 0u;
            if (alive && (tagged >> 8) != ((uint32_t)k & 0xffffffu)) {
                if (lane == 0) {
                    atomicOr(p.err, SHKV_ERRF_PIPELINE);
                    *c.abort_flag = 1u;
                }
                alive = false;
            }
            const uint32_t mask = tagged & 0xffu;
            const int tok0 = s.p0 * P + j * TT;
            const bool all_valid = (mask == (1u << (TT / BR)) - 1u) && (tok0 + TT <= lim);
            auto tok_valid = [&](int t) -> bool { return ((mask >> (t >> log2BR)) & 1u) && (tok0 + t < lim); };
            if (alive && !all_valid && warp == 0) {
                // masked V rows may hold stale or non-finite bits: zero them
                const uint32_t vst = c.lay.ring + (uint32_t)slot * c.lay.stage_bytes + (uint32_t)(TT * D * 2);
                for (int e = lane; e < TT * (D / 8); e += 32) {
                    const int t = e / (D / 8);
                    const int ch = e - t * (D / 8);
                    if (!tok_valid(t))
                        *reinterpret_cast<uint4 *>(c.smem + vst + (uint32_t)((t >> log2BR) * (BR * D * 2) +
                                                                                (ch >> 3) * (BR * 128) +
                                                                                (t & (BR - 1)) * 128 + (ch & 7) * 16)) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
            }
            // --- masked, scaled scores and the tile max (base 2)
            float xs[32];
            float mt = -INFINITY;
#pragma unroll
            for (int t = 0; t < 32; ++t) {
                float v = __uint_as_float(sv[t]) * sl2;
                if (!all_valid && !tok_valid(t))
                    v = -INFINITY;
                xs[t] = v;
                mt = fmaxf(mt, v);
            }
            // --- lazy rescale of this row's O when its max jumps by > 2^8
            const bool need = alive && m_use != -INFINITY && mt > m_use + kRescaleLog2;
            if (__any_sync(0xffffffffu, need) && alive && j >= 1) {
                // O must hold PV of the previous stage before it is touched
                wait(p_free_bar(x, (k - 1) & 1), (uint32_t)(((k - 1) >> 1) & 1));
                if (alive) {
                    tc_fence_after();
                    const float alpha = need ? ex2_approx(m_use - mt) : 1.f;
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        uint32_t ov[32];
                        tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(cc * 32), ov);
#pragma unroll
                        for (int t = 0; t < 32; ++t)
                            ov[t] = __float_as_uint(__uint_as_float(ov[t]) * alpha);
                        tmem_st32(tmem + lane_base + kTmemO + (uint32_t)(cc * 32), ov);
                    }
                    tc_fence_before();
                    if (need) {
                        lsum *= alpha;
                        m_use = mt;
                    }
                }
            }
            if (m_use == -INFINITY)
                m_use = mt;                      // first scored tile of the segment
            const float mu = m_use == -INFINITY ? 0.f : m_use;
            uint32_t pk[16];
#pragma unroll
            for (int t = 0; t < 32; t += 2) {
                const float p0 = ex2_approx(xs[t] - mu);
                const float p1 = ex2_approx(xs[t + 1] - mu);
                lsum += p0 + p1;
                pk[t / 2] = pack_bf16x2(p0, p1);
            }
            // --- this row of P into the tile of this stage's parity
            wait(p_free_bar(x, buf), (uint32_t)(((k >> 1) & 1) ^ 1));
            if (alive && active) {
                const uint32_t prow = ptile(x, buf) - c.base + (uint32_t)r * 128u;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    *reinterpret_cast<uint4 *>(c.smem + prow + (uint32_t)((ch ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(p_full_bar(x, buf));
        }

        // --- segment end: this row of O, normalised
        const int last = kbase + nst - 1;
        wait(p_free_bar(x, last & 1), (uint32_t)((last >> 1) & 1));
        const bool whole = (s.seg_begin == s.unit_begin) && (s.seg_end == s.unit_end);
        const int slot_id = whole ? 0 : 2 * (int)blockIdx.x + (s.seg_begin == c.cta_begin ? 0 : 1);
        const float inv = lsum > 0.f ? __frcp_rn(lsum) : 0.f;
        const int64_t orow = whole ? (int64_t)s.b * p.n_models * p.hq + q_row(p, s.g, active ? r : 0)
                                   : (int64_t)slot_id * p.rows + r;
        if (alive)
            tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t ov[32];
            if (alive)
                tmem_ld32(tmem + lane_base + kTmemO + (uint32_t)(cc * 32), ov);
            if (alive && active) {
                if (whole) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + cc * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(ov[q4 * 8 + 2 * e]) * inv,
                                               __uint_as_float(ov[q4 * 8 + 2 * e + 1]) * inv);
                        dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(p.ws_part + orow * D + cc * 32);
#pragma unroll
                    for (int q4 = 0; q4 < 8; ++q4)
                        dst[q4] = make_float4(__uint_as_float(ov[4 * q4]) * inv, __uint_as_float(ov[4 * q4 + 1]) * inv,
                                              __uint_as_float(ov[4 * q4 + 2]) * inv,
                                              __uint_as_float(ov[4 * q4 + 3]) * inv);
                }
            }
        }
        tc_fence_before();
        if (alive && active) {
            const float lse = lsum > 0.f ? (m_use + log2f(lsum)) * kLn2u : -INFINITY;
            if (whole) {
                if (p.lse_out)
                    p.lse_out[orow] = lse;
            } else {
                p.ws_lse[orow] = lse;
            }
        }
        named_barrier(1, 32u * kSoftmaxWarps);

        // --- split unit: the last piece to arrive merges all pieces
        if (!whole) {
            const int c0 = cta_of(p, s.unit_begin);
            const int c1 = cta_of(p, s.unit_end - 1);
            uint32_t *counter = p.ws_count + (int64_t)s.b * p.hkv + s.g;
            if (threadIdx.x == 0) {
                __threadfence();
                const uint32_t prev = atomicAdd(counter, 1u);
                *c.bcast = (prev == (uint32_t)(c1 - c0)) ? 1u : 0u;
            }
            named_barrier(1, 32u * kSoftmaxWarps);
            if (*c.bcast) {
                __threadfence();
                const int dq = D / 4;
                for (int rr = warp; rr < p.rows; rr += kSoftmaxWarps) {
                    float M = -INFINITY;
                    for (int cc = c0 + lane; cc <= c1; cc += 32)
                        M = fmaxf(M, __ldcg(p.ws_lse + (int64_t)piece_slot(p, cc, s.unit_begin) * p.rows + rr));
#pragma unroll
                    for (int o_ = 16; o_ > 0; o_ >>= 1)
                        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o_));
                    float wsum = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (M != -INFINITY) {
                        for (int cc = c0; cc <= c1; ++cc) {
                            const int sl = piece_slot(p, cc, s.unit_begin);
                            const float w = ex2_approx((__ldcg(p.ws_lse + (int64_t)sl * p.rows + rr) - M) *
                                                       1.4426950408889634f);
                            wsum += w;
                            if (lane < dq) {
                                const float4 v = __ldcg(reinterpret_cast<const float4 *>(
                                                            p.ws_part + ((int64_t)sl * p.rows + rr) * D) + lane);
                                acc.x += w * v.x;
                                acc.y += w * v.y;
                                acc.z += w * v.z;
                                acc.w += w * v.w;
                            }
                        }
                    }
                    const float winv = wsum > 0.f ? 1.f / wsum : 0.f;
                    const int64_t orr = (int64_t)s.b * p.n_models * p.hq + q_row(p, s.g, rr);
                    if (lane < dq) {
                        uint2 packed;
                        packed.x = pack_bf16x2(acc.x * winv, acc.y * winv);
                        packed.y = pack_bf16x2(acc.z * winv, acc.w * winv);
                        *reinterpret_cast<uint2 *>(p.out + orr * D + lane * 4) = packed;
                    }
                    if (lane == 0 && p.lse_out)
                        p.lse_out[orr] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
                }
                if (threadIdx.x == 0)
                    *counter = 0u;
            }
            named_barrier(1, 32u * kSoftmaxWarps);
        }

        kbase += nst;
        ++seg;
        if (s.seg_end >= c.cta_end)
            break;
        s = next_segment(p, s, c.cta_end);
    }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kUmmaThreads, 1)
    shkv_decode_umma_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                            const __grid_constant__ DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    UCtx x;
    Ctx &c = x.c;
    {
        const uint32_t raw = smem_u32(smem_raw);
        const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
        c.smem = smem_raw + pad;
        c.base = raw + pad;
    }
    x.u = umma_smem_layout(D, p.rows, p.stages);
    c.lay = x.u.s;
    c.abort_flag = reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.misc);
    c.bcast = reinterpret_cast<uint32_t *>(c.smem + c.lay.misc + 4);
    c.cta_begin = p.cta_cut[blockIdx.x];
    c.cta_end = p.cta_cut[blockIdx.x + 1];
    const int warp = threadIdx.x >> 5;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full_bar(c, s), 1);
            mbar_init(empty_bar(c, s, p.stages), 1);         // one tcgen05.commit per stage
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull_bar(c, i, p.stages), 1);
            mbar_init(qempty_bar(c, i, p.stages), kSoftmaxWarps);
            mbar_init(s_full_bar(x, i), 1);
            mbar_init(s_free_bar(x, i), kSoftmaxWarps);
            mbar_init(p_full_bar(x, i), kSoftmaxWarps);
            mbar_init(p_free_bar(x, i), 1);
        }
        mbar_init(q_ready_bar(x), kSoftmaxWarps);
        mbar_init(q_tile_free_bar(x), 1);
        mbar_init(fin_bar(x), 1);
        *c.abort_flag = 0u;
        *c.bcast = 0u;
        fence_barrier_init();
    }
    if (warp == 0)
        tmem_alloc(c.base + x.u.tslot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(c.smem + x.u.tslot);

    if (warp == kProducerWarp)
        producer<D>(&tmK, &tmV, p, c);
    else if (warp == kMmaWarp) {
        if ((threadIdx.x & 31) == 0)
            mma_issuer<D>(p, x, tmem);
    } else
        softmax_rows<D>(p, x, tmem);

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
uint32_t umma_smem_bytes(int D, int rows, int stages) { return umma_smem_layout(D, rows, stages).s.total; }

template <int D>
static cudaError_t launch_umma_t(const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p,
                                 uint32_t smem, cudaStream_t stream)
{
    auto kern = shkv_decode_umma_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    kern<<<p.num_ctas, kUmmaThreads, smem, stream>>>(tmK, tmV, p);
    return cudaGetLastError();
}

cudaError_t launch_decode_umma(int D, const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p,
                               uint32_t smem, cudaStream_t stream)
{
    return D == 128 ? launch_umma_t<128>(tmK, tmV, p, smem, stream) : launch_umma_t<64>(tmK, tmV, p, smem, stream);
}

}  // namespace shkv
