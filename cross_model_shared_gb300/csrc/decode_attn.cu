// decode_attn.cu -- shared-KV multi-decoder paged decode attention (sm_103a).
//
// The method (ICaRus, key design 3; PrefillShare Sec. 3.3): N decoders that
// share one frozen encoder also share one paged KV cache, and their queries
// are stacked along the head axis so that all of them attend the cache
// together.  For KV head g the stacked rows are the R = N * (Hq / Hkv) query
// heads of every decoder that map to g; each K/V page of head g is therefore
// fetched from HBM once per step and applied to all R rows while it sits in
// shared memory.  Decode is memory-bound (PrefillShare Sec. 4, two-phase
// execution), so the R-fold reuse is what hides the extra decoders' compute.
//
// Work decomposition (flash-decoding with a balanced static split):
//   The (request b, KV head g, page p) chunks, ordered request-major, are cut
//   into num_ctas contiguous ranges of equal cost (chunks plus a fixed cost
//   per segment, planned on the host); one persistent CTA per SM walks its
//   range as a sequence of segments (one segment per (b, g) it touches).  A
//   (b, g) that straddles a cut is split: each piece writes a normalised
//   partial and its log-sum-exp, and the last piece to finish (an atomic
//   arrival counter, no waiting) merges them; a piece that reads, early in
//   its epilogue, that every other piece has arrived merges without
//   arriving.  No CTA ever waits for another.
//
// Launches are chained by programmatic dependent launch; before waiting for
// the previous launch the producer prefetches its first ring-full of pages
// into L2 (prefetches only: nothing read before the wait is used after it).
//
// Inside a CTA:
//   * one producer warp streams K and V into an mbarrier ring of
//     kStageTokens-token slots.  Each copy is one 3-D TMA box covering a whole
//     row-block of one head's page (4 or 8 KiB, 128-byte swizzle, L2
//     evict-first), and the copies of a slot are issued by several lanes in
//     one instruction: a single thread issuing small copies one at a time
//     cannot keep HBM busy.  A bulk copy brings the segment's R query rows;
//     block-table entries are prefetched 32 at a time;
//   * consumer warps take slots round-robin, fewer warps than slots so most
//     of the ring stays in flight.  Each warp owns 8 or 16 stacked rows (a
//     row group); larger R uses several row groups that read the same slot.  Per slot a warp computes S^T = K Q^T with tokens as the MMA M
//     dimension (16 tokens x 8 rows per mma.sync m16n8k16), so R = 8 rows fill
//     an MMA exactly; an online softmax in base 2 follows; P^T is transposed in
//     registers (movmatrix) and O^T += V^T P^T accumulates in fp32;
//   * at the end of a segment the warps of a row group merge their
//     (max, sum, O) states through shared memory; each warp then combines
//     and writes its own share of the accumulator registers.
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

// ---------------------------------------------------------------------------
// consumer warps
// ---------------------------------------------------------------------------
template <int D, int NT, bool FUSED>
__device__ void consumer(const DecodeParams &p, const Ctx &c)
{
    constexpr int KSTEPS = D / 16;
    constexpr int ROWS_W = 8 * NT;
    constexpr int NREG = KSTEPS * NT * 4;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ncw = p.nrg * p.wt;
    const int rg = warp / p.wt;
    const int wtid = warp - rg * p.wt;
    const int row0 = rg * ROWS_W;
    const int stages = p.stages;
    constexpr int TT = kStageTokens;
    constexpr int MTS = TT / 16;                   // 16-token MMA tiles per stage
    const int P = p.page_size;
    const int BR = p.box_rows;
    const int log2BR = 31 - __clz(BR);
    const float sl2 = p.scale_log2;
    // Stage layout: [row-block][column half][row][128 bytes], swizzled per 8 rows.
    auto row_off = [&](int t) -> uint32_t {
        return (uint32_t)((t >> log2BR) * (BR * D * 2) + (t & (BR - 1)) * 128);
    };

    float *comb_o = reinterpret_cast<float *>(c.smem + c.lay.comb_o);
    float *comb_m = reinterpret_cast<float *>(c.smem + c.lay.comb_m);
    float *comb_l = reinterpret_cast<float *>(c.smem + c.lay.comb_l);
    const volatile uint32_t *meta = reinterpret_cast<const volatile uint32_t *>(c.smem + c.lay.meta);

    // per-lane constant parts of the ldmatrix addresses
    const int k_tok = (lane & 7) + ((lane >> 3) & 1) * 8;   // K: token within a 16-token tile
    const int k_col = (lane >> 4) * 8;                        // K: column offset within 16
    const int v_tok = (lane & 7) + ((lane >> 4) & 1) * 8;   // V: token within a 16-token tile
    const int v_col = ((lane >> 3) & 1) * 8;                  // V: column offset within 16

    // output row of this lane's rows (nt, i) without the KV head's term g*G:
    // fixed for the whole launch
    int qoff[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int r = row0 + nt * 8 + 2 * (lane & 3) + i;
            qoff[nt][i] = q_row(p, 0, r < p.rows ? r : 0);
        }

    bool alive = true;
    int kbase = 0, seg = 0;
    Segment s = locate(p, c.cta_begin, c.cta_end);
    for (;;) {
        const int tok_end = s.p1 * P;
        const int nst = (tok_end - s.p0 * P + TT - 1) / TT;
        const int qb = seg & 1;

        // --- query fragments (B operand of S^T = K Q^T): rows row0.., all D
        uint32_t qf[KSTEPS][NT][2];
        {
            bool ok = true;
            if (alive) {
                ok = mbar_wait_bounded(qfull_bar(c, qb, stages), (seg >> 1) & 1, c.abort_flag, p.err);
                alive = __all_sync(0xffffffffu, ok);
            }
            const uint32_t qbase = c.base + c.lay.qbuf + qb * c.lay.qbuf_bytes;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ks += 2) {
                    const uint32_t addr = qbase + (uint32_t)((row0 + nt * 8 + (lane & 7)) * D * 2) +
                                          (uint32_t)((ks * 16 + (lane >> 3) * 8) * 2);
                    if (alive)
                        ldsm_x4(addr, qf[ks][nt][0], qf[ks][nt][1], qf[ks + 1][nt][0], qf[ks + 1][nt][1]);
                    else
                        qf[ks][nt][0] = qf[ks][nt][1] = qf[ks + 1][nt][0] = qf[ks + 1][nt][1] = 0u;
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(qempty_bar(c, qb, stages));
        }

        // --- cached length, from the plan (the producer checks the device copy);
        // fused tails take each page's valid tokens from page_info instead
        constexpr bool fused = FUSED;
        const int L = fused ? tok_end : plan_len(p, s);
        const int lim = L < tok_end ? L : tok_end;     // tokens of this segment that count

        float o[KSTEPS][NT][4];
        float mrow[NT][2], lrow[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            mrow[nt][0] = mrow[nt][1] = -INFINITY;
            lrow[nt][0] = lrow[nt][1] = 0.f;
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt)
                o[mt][nt][0] = o[mt][nt][1] = o[mt][nt][2] = o[mt][nt][3] = 0.f;
        }

        for (int j = (wtid - kbase % p.wt + p.wt) % p.wt; j < nst; j += p.wt) {
            const int k = kbase + j;
            const int slot = k % stages;
            bool ok = false;
            if (alive) {
                ok = mbar_wait_bounded(full_bar(c, slot), (k / stages) & 1, c.abort_flag, p.err);
                ok = __all_sync(0xffffffffu, ok);
                alive = ok;
            }
            bool tag_ok = true;
            if (ok && (meta[slot * kMetaWords] >> 8) != ((uint32_t)k & 0xffffffu)) {
                // The slot holds another stage: report it, stop this CTA
                // (bounded) and do not arrive, so no copy is re-armed over it.
                tag_ok = false;
                ok = false;
                alive = false;
                if (lane == 0) {
                    atomicOr(p.err, SHKV_ERRF_PIPELINE);
                    *c.abort_flag = 1u;
                }
            }
            if (ok) {
                const uint32_t kst = c.base + c.lay.ring + (uint32_t)slot * c.lay.stage_bytes;
                const uint32_t vst = kst + (uint32_t)(TT * D * 2);
                const uint32_t mask = meta[slot * kMetaWords] & 0xffu;
                const int tok0 = s.p0 * P + j * TT;       // logical token of slot row 0
                const uint32_t full_mask = (1u << (TT / BR)) - 1u;
                // fused tails: per row-block (one page) its valid tokens and
                // the decoder whose rows attend it
                const uint32_t whole = kAllDecoders << 8 | (uint32_t)BR;
                uint32_t inf0 = whole, inf1 = whole;
                if (fused) {
                    inf0 = meta[slot * kMetaWords + 1];
                    inf1 = TT / BR > 1 ? meta[slot * kMetaWords + 2] : inf0;
                }
                // every token of the stage is a real key (no V row to clear) ...
                const bool toks_valid =
                    (mask == full_mask) &&
                    (fused ? ((inf0 & 0xffu) == (uint32_t)BR && (inf1 & 0xffu) == (uint32_t)BR) : (tok0 + TT <= lim));
                // ... and every row attends every token (no score to mask)
                const bool all_valid = toks_valid && (!fused || (inf0 == whole && inf1 == whole));
                auto tok_valid = [&](int t) -> bool {
                    if (!fused)
                        return ((mask >> (t >> log2BR)) & 1u) && (tok0 + t < lim);
                    const int rb = t >> log2BR;
                    return ((mask >> rb) & 1u) && (uint32_t)(t & (BR - 1)) < ((rb ? inf1 : inf0) & 0xffu);
                };
                // (fused tails) row r of the N*G stacked rows attends token t
                auto row_attends = [&](int t, int r) -> bool {
                    const uint32_t dec = (((t >> log2BR) ? inf1 : inf0) >> 8) & 0xffu;
                    return dec == kAllDecoders || (uint32_t)(r - (int)dec * p.group) < (uint32_t)p.group;
                };
                if (!toks_valid) {
                    // Rows that are masked may hold stale or non-finite bits:
                    // zero their V so 0 * V stays 0 in the PV product.
                    for (int e = lane; e < TT * (D / 8); e += 32) {
                        const int t = e / (D / 8);
                        const int cchunk = e - t * (D / 8);
                        if (!tok_valid(t))
                            st_shared_zero16(vst + row_off(t) + (uint32_t)((cchunk >> 3) * (BR * 128) + (cchunk & 7) * 16));
                    }
                    __syncwarp();
                }

                // S^T[tok, row] = K[tok, :] . Q[row, :]; even and odd k-steps
                // accumulate separately to halve the dependent MMA chain.
                float sc[MTS][NT][4], sc2[MTS][NT][4];
#pragma unroll
                for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            sc[mt][nt][e] = sc2[mt][nt][e] = 0.f;
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
                    for (int mt = 0; mt < MTS; ++mt) {
                        const int tok = mt * 16 + k_tok;
                        const int col = ks * 16 + k_col;
                        const uint32_t addr = kst + row_off(tok) + (uint32_t)((col >> 6) * (BR * 128) +
                                                                            ((((col & 63) >> 3) ^ (tok & 7)) << 4));
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(addr, a0, a1, a2, a3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_bf16((ks & 1) ? sc2[mt][nt] : sc[mt][nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
                    }
                }

                // online softmax in base 2: x = s * scale * log2(e)
#pragma unroll
                for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            float x = (sc[mt][nt][e] + sc2[mt][nt][e]) * sl2;
                            if (!all_valid) {
                                const int tt = mt * 16 + (lane >> 2) + (e >> 1) * 8;
                                if (!tok_valid(tt) ||
                                    (fused && !row_attends(tt, row0 + nt * 8 + (lane & 3) * 2 + (e & 1))))
                                    x = -INFINITY;
                            }
                            sc[mt][nt][e] = x;
                        }
                uint32_t pb[MTS][NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float mx[2];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        float v = fmaxf(sc[0][nt][i], sc[0][nt][i + 2]);
#pragma unroll
                        for (int mt = 1; mt < MTS; ++mt)
                            v = fmaxf(v, fmaxf(sc[mt][nt][i], sc[mt][nt][i + 2]));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                        mx[i] = v;
                    }
                    float alpha[2], muse[2];
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const float mnew = fmaxf(mrow[nt][i], mx[i]);
                        muse[i] = (mnew == -INFINITY) ? 0.f : mnew;
                        alpha[i] = ex2_approx(mrow[nt][i] - muse[i]);
                        mrow[nt][i] = mnew;
                    }
                    float rs[2] = {0.f, 0.f};
#pragma unroll
                    for (int mt = 0; mt < MTS; ++mt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float pv = ex2_approx(sc[mt][nt][e] - muse[e & 1]);
                            sc[mt][nt][e] = pv;
                            rs[e & 1] += pv;
                        }
                    lrow[nt][0] = lrow[nt][0] * alpha[0] + rs[0];
                    lrow[nt][1] = lrow[nt][1] * alpha[1] + rs[1];
                    // rescale O only if some row's running max moved
                    if (!__all_sync(0xffffffffu, alpha[0] == 1.f && alpha[1] == 1.f)) {
#pragma unroll
                        for (int mt = 0; mt < KSTEPS; ++mt) {
                            o[mt][nt][0] *= alpha[0];
                            o[mt][nt][1] *= alpha[1];
                            o[mt][nt][2] *= alpha[0];
                            o[mt][nt][3] *= alpha[1];
                        }
                    }
#pragma unroll
                    for (int kt = 0; kt < MTS; ++kt) {
                        pb[kt][nt][0] = movmatrix_trans(pack_bf16x2(sc[kt][nt][0], sc[kt][nt][1]));
                        pb[kt][nt][1] = movmatrix_trans(pack_bf16x2(sc[kt][nt][2], sc[kt][nt][3]));
                    }
                }

                // O^T[d, row] += V^T[d, tok] . P^T[tok, row]
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
#pragma unroll
                    for (int kt = 0; kt < MTS; ++kt) {
                        const int tok = kt * 16 + v_tok;
                        const int col = mt * 16 + v_col;
                        const uint32_t addr = vst + row_off(tok) + (uint32_t)((col >> 6) * (BR * 128) +
                                                                            ((((col & 63) >> 3) ^ (tok & 7)) << 4));
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_t(addr, a0, a1, a2, a3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_bf16(o[mt][nt], a0, a1, a2, a3, pb[kt][nt][0], pb[kt][nt][1]);
                    }
                }
                if (!toks_valid)
                    fence_proxy_async_smem();   // generic zero-writes before the next TMA into this slot
            }
            __syncwarp();
            if (lane == 0 && tag_ok)
                mbar_arrive(empty_bar(c, slot, stages));
        }

        // A split piece's unit count, read now so that its latency hides behind
        // the epilogue: when every other piece has arrived already, this one
        // merges without arriving (see below).
        uint32_t pre_count = 0xffffffffu;
        if (threadIdx.x == 0 && !(s.seg_begin == s.unit_begin && s.seg_end == s.unit_end))
            pre_count = ld_acquire_gpu(p.ws_count + (int64_t)s.b * p.hkv + s.g);

        // --- merge the row group's warps: publish (m, l, O) ...
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                float v = lrow[nt][i];
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                v += __shfl_xor_sync(0xffffffffu, v, 8);
                v += __shfl_xor_sync(0xffffffffu, v, 16);
                lrow[nt][i] = v;
            }
        if (lane < 4) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    comb_m[warp * ROWS_W + nt * 8 + 2 * lane + i] = mrow[nt][i];
                    comb_l[warp * ROWS_W + nt * 8 + 2 * lane + i] = lrow[nt][i];
                }
        }
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    comb_o[((size_t)warp * NREG + (mt * NT + nt) * 4 + e) * 32 + lane] = o[mt][nt][e];
        named_barrier(1, (uint32_t)ncw * 32u);

        // ... then combine them.  Each lane first derives, for the 2*NT rows
        // its registers touch, the factor exp2(m_w - M) / L of every warp w
        // of the group; every element is then one FMA per warp.
        const bool whole = (s.seg_begin == s.unit_begin) && (s.seg_end == s.unit_end);
        const int slot_id = whole ? 0 : 2 * (int)blockIdx.x + (s.seg_begin == c.cta_begin ? 0 : 1);
        const int w_first = rg * p.wt;
        float fac[NT][2][kWtMax];
        int64_t orow_r[NT][2];
        const int64_t rbase = whole ? (int64_t)s.b * p.n_models * p.hq + (int64_t)s.g * p.group
                                    : (int64_t)slot_id * p.rows;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int rl = nt * 8 + 2 * (lane & 3) + i;
                // every warp's (m, l) of this row first, so the loads issue together
                float mw[kWtMax], lw[kWtMax];
#pragma unroll
                for (int w = 0; w < kWtMax; ++w) {
                    mw[w] = w < p.wt ? comb_m[(w_first + w) * ROWS_W + rl] : -INFINITY;
                    lw[w] = w < p.wt ? comb_l[(w_first + w) * ROWS_W + rl] : 0.f;
                }
                float M = -INFINITY;
#pragma unroll
                for (int w = 0; w < kWtMax; ++w)
                    if (w < p.wt)
                        M = fmaxf(M, mw[w]);
                float lsum = 0.f;
#pragma unroll
                for (int w = 0; w < kWtMax; ++w) {
                    fac[nt][i][w] = 0.f;
                    if (w < p.wt && M != -INFINITY) {
                        fac[nt][i][w] = ex2_approx(mw[w] - M);
                        lsum += lw[w] * fac[nt][i][w];
                    }
                }
                const float inv = lsum > 0.f ? __frcp_rn(lsum) : 0.f;
#pragma unroll
                for (int w = 0; w < kWtMax; ++w)
                    fac[nt][i][w] *= inv;
                const int r = row0 + rl;
                orow_r[nt][i] = rbase + (whole ? (int64_t)qoff[nt][i] : (int64_t)r);
                if (wtid == 0 && (lane >> 2) == 0 && r < p.rows) {     // one writer per row
                    const float lse = lsum > 0.f ? (M + log2f(lsum)) * kLn2 : -INFINITY;
                    if (whole) {
                        if (p.lse_out)
                            p.lse_out[orow_r[nt][i]] = lse;
                    } else {
                        p.ws_lse[orow_r[nt][i]] = lse;
                    }
                }
            }
        // element (mt, nt, e) is register reg = (mt*NT + nt)*4 + e of the row
        // group's O; warp wtid of the group takes the registers with
        // reg % wt == wtid.  A loop over just those, unrolled, so the shared
        // memory loads of several elements are in flight together (this runs
        // once per segment on one warp per SM sub-partition: latency-bound).
#pragma unroll 8
        for (int reg = wtid; reg < NREG; reg += p.wt) {
            const int e = reg & 3, i = e & 1;
            const int nt = NT > 1 ? (reg >> 2) % NT : 0;
            const int mt = (reg >> 2) / NT;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < kWtMax; ++w)
                if (w < p.wt) {
                    const float f = (NT > 1 && nt) ? (i ? fac[NT - 1][1][w] : fac[NT - 1][0][w])
                                                   : (i ? fac[0][1][w] : fac[0][0][w]);
                    acc += comb_o[((size_t)(w_first + w) * NREG + reg) * 32 + lane] * f;
                }
            const int r = row0 + nt * 8 + 2 * (lane & 3) + i;
            if (r < p.rows) {
                const int64_t orow = (NT > 1 && nt) ? (i ? orow_r[NT - 1][1] : orow_r[NT - 1][0])
                                                    : (i ? orow_r[0][1] : orow_r[0][0]);
                const int d = mt * 16 + (lane >> 2) + (e >> 1) * 8;
                if (!whole)
                    p.ws_part[orow * D + d] = acc;
                else
                    p.out[orow * D + d] = __float2bfloat16_rn(acc);
            }
        }
        named_barrier(1, (uint32_t)ncw * 32u);

        // --- split unit: the last piece to arrive merges all pieces
        if (!whole) {
            const int c0 = cta_of(p, s.unit_begin);
            const int c1 = cta_of(p, s.unit_end - 1);
            uint32_t *counter = p.ws_count + (int64_t)s.b * p.hkv + s.g;
            if (threadIdx.x == 0) {
                if (pre_count == (uint32_t)(c1 - c0)) {
                    // every other piece had arrived (acquire read above): this is
                    // the last one, so it merges without arriving
                    *c.bcast = 1u;
                } else {
                    __threadfence();     // this CTA's partial (ordered by the barrier above) before the count
                    const uint32_t prev = atomicAdd(counter, 1u);
                    *c.bcast = (prev == (uint32_t)(c1 - c0)) ? 1u : 0u;
                }
            }
            named_barrier(1, (uint32_t)ncw * 32u);
            if (*c.bcast) {
                __threadfence();
                // one warp per stacked row: the split log-sum-exps, then the
                // weighted sum of the split outputs, loads issued together
                const int dq = D / 4;
                for (int r = warp; r < p.rows; r += ncw) {
                    float M = -INFINITY;
                    for (int cc = c0 + lane; cc <= c1; cc += 32)
                        M = fmaxf(M, __ldcg(p.ws_lse + (int64_t)piece_slot(p, cc, s.unit_begin) * p.rows + r));
#pragma unroll
                    for (int o_ = 16; o_ > 0; o_ >>= 1)
                        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o_));
                    float wsum = 0.f;
                    float4 acc[D / 128 > 0 ? D / 128 : 1];
#pragma unroll
                    for (int h = 0; h < (D / 128 > 0 ? D / 128 : 1); ++h)
                        acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (M != -INFINITY) {
                        for (int cc = c0; cc <= c1; ++cc) {
                            const int sl = piece_slot(p, cc, s.unit_begin);
                            const float w = ex2_approx((__ldcg(p.ws_lse + (int64_t)sl * p.rows + r) - M) *
                                                       1.4426950408889634f);
                            wsum += w;
                            const float4 *src = reinterpret_cast<const float4 *>(p.ws_part + ((int64_t)sl * p.rows + r) * D);
#pragma unroll
                            for (int h = 0; h < (D / 128 > 0 ? D / 128 : 1); ++h) {
                                const int d4 = lane + 32 * h;
                                if (d4 < dq) {
                                    const float4 v = __ldcg(src + d4);
                                    acc[h].x += w * v.x;
                                    acc[h].y += w * v.y;
                                    acc[h].z += w * v.z;
                                    acc[h].w += w * v.w;
                                }
                            }
                        }
                    }
                    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
                    const int64_t orow = (int64_t)s.b * p.n_models * p.hq + q_row(p, s.g, r);
#pragma unroll
                    for (int h = 0; h < (D / 128 > 0 ? D / 128 : 1); ++h) {
                        const int d4 = lane + 32 * h;
                        if (d4 < dq) {
                            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[h].x * inv, acc[h].y * inv);
                            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[h].z * inv, acc[h].w * inv);
                            uint2 packed;
                            packed.x = *reinterpret_cast<uint32_t *>(&lo);
                            packed.y = *reinterpret_cast<uint32_t *>(&hi);
                            *reinterpret_cast<uint2 *>(p.out + orow * D + d4 * 4) = packed;
                        }
                    }
                    if (lane == 0 && p.lse_out)
                        p.lse_out[orow] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
                }
                if (threadIdx.x == 0)
                    *counter = 0u;
            }
            named_barrier(1, (uint32_t)ncw * 32u);
        }

        kbase += nst;
        ++seg;
        if (s.seg_end >= c.cta_end)
            break;
        s = next_segment(p, s, c.cta_end);
    }
}

}  // namespace

// FUSED: the units are fused per-decoder tails (DecodeParams::page_info).
template <int D, int NT, bool FUSED>
__global__ void __launch_bounds__(NT == 1 ? kMaxThreadsNT1 : kMaxThreadsNT2, 1)
    shkv_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const __grid_constant__ DecodeParams p)
{
    extern __shared__ uint8_t smem_raw[];
    Ctx c;
    {
        const uint32_t raw = smem_u32(smem_raw);
        const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
        c.smem = smem_raw + pad;
        c.base = raw + pad;
    }
    constexpr int KSTEPS = D / 16;
    const int ncw = p.nrg * p.wt;
    c.lay = decode_smem_layout(D, 8 * NT, KSTEPS * NT * 4, ncw, p.rpad, p.stages);
    c.abort_flag = reinterpret_cast<volatile uint32_t *>(c.smem + c.lay.misc);
    c.bcast = reinterpret_cast<uint32_t *>(c.smem + c.lay.misc + 4);
    c.cta_begin = p.cta_cut[blockIdx.x];
    c.cta_end = p.cta_cut[blockIdx.x + 1];

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full_bar(c, s), 1);
            mbar_init(empty_bar(c, s, p.stages), (uint32_t)p.nrg);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(qfull_bar(c, i, p.stages), 1);
            mbar_init(qempty_bar(c, i, p.stages), (uint32_t)ncw);
        }
        *c.abort_flag = 0u;
        *c.bcast = 0u;
        fence_barrier_init();
    }
    // rows [R, rpad) of both query buffers are padding: zero them once
    {
        const int pad_rows = p.rpad - p.rows;
        const int n16 = pad_rows * D * 2 / 16;
        for (int i = threadIdx.x; i < 2 * n16; i += blockDim.x) {
            const int bufi = i / (n16 > 0 ? n16 : 1);
            const int e = i - bufi * n16;
            st_shared_zero16(c.base + c.lay.qbuf + bufi * c.lay.qbuf_bytes + p.rows * D * 2 + e * 16);
        }
    }
    fence_proxy_async_smem();
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    if (warp == ncw) {
        warm_l2<D>(&tmK, &tmV, p, c);
        pdl_wait_prior();                   // global memory only from here on
        pdl_launch_dependents();            // (after the wait: see launch.cuh)
        producer<D, FUSED>(&tmK, &tmV, p, c);
    } else {
        pdl_wait_prior();
        pdl_launch_dependents();
        if (warp < ncw)
            consumer<D, NT, FUSED>(p, c);
    }
}

// ---------------------------------------------------------------------------
// host-side launcher (internal to the library)
// ---------------------------------------------------------------------------
template <int D, int NT, bool FUSED>
static cudaError_t launch_decode_f(const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p,
                                   uint32_t smem, cudaStream_t stream)
{
    auto kern = shkv_decode_kernel<D, NT, FUSED>;
    static uint32_t configured = 0;
    if (smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        configured = smem;
    }
    const int threads = (p.nrg * p.wt + 1) * 32;
    return launch_pdl(kern, p.num_ctas, threads, smem, stream, tmK, tmV, p);
}

template <int D, int NT>
static cudaError_t launch_decode_t(const CUtensorMap &tmK, const CUtensorMap &tmV, const DecodeParams &p,
                                   uint32_t smem, cudaStream_t stream)
{
    return p.fused ? launch_decode_f<D, NT, true>(tmK, tmV, p, smem, stream)
                   : launch_decode_f<D, NT, false>(tmK, tmV, p, smem, stream);
}

cudaError_t launch_decode(int D, int NT, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          const DecodeParams &p, uint32_t smem, cudaStream_t stream)
{
    if (D == 128)
        return NT == 1 ? launch_decode_t<128, 1>(tmK, tmV, p, smem, stream)
                       : launch_decode_t<128, 2>(tmK, tmV, p, smem, stream);
    return NT == 1 ? launch_decode_t<64, 1>(tmK, tmV, p, smem, stream)
                   : launch_decode_t<64, 2>(tmK, tmV, p, smem, stream);
}

}  // namespace shkv
