// append_merge.cu -- partial-prefill append and the split-KV merge (sm_103a).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "launch.cuh"
#include "shkv_device.cuh"
#include "tails.cuh"

namespace shkv {

// Partial-prefill append (PrefillShare Sec. 3.3 / Sec. 7): token t of request
// b lands at logical position L_b + t of the shared paged cache.  One warp
// per appended token: its page and slot are looked up once, then the lanes
// move the token's Hkv head rows of K and V (D bf16 each) as 16-byte vectors
// -- contiguous on the source side, whole head rows of 128 or 256 bytes on
// the destination side.  The old lengths come from the pool's host copy;
// block 0 then publishes L_b + T (no thread of this kernel reads seq_lens
// after that store).
__global__ void __launch_bounds__(256) shkv_append_kernel(const __grid_constant__ AppendParams p)
{
    pdl_wait_prior();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int hv = p.head_vecs;                      // 16-byte vectors per head row: 8 or 16
    const int log2hv = __ffs(hv) - 1;
    const int per_tok = p.hkv * hv;                  // vectors per token, of K or of V
    const int64_t ntok = (int64_t)p.batch * p.n_new;
    for (int64_t tok = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); tok < ntok;
         tok += (int64_t)gridDim.x * warps) {
        const int b = (int)(tok / p.n_new);
        const int t = (int)(tok - (int64_t)b * p.n_new);
        const int pos = p.old_len[b] + t;
        const int page = __ldg(p.block_table + (int64_t)b * p.max_pages + pos / p.page_size);
        if (page < 0 || page >= p.num_pages) {
            if (lane == 0)
                atomicOr(p.err, SHKV_ERRF_PAGE_OOB);
            continue;
        }
        const int slot = pos % p.page_size;
        const uint4 *ks = p.k_new + tok * per_tok;
        const uint4 *vs = p.v_new + tok * per_tok;
        const int64_t row0 = (int64_t)page * p.hkv;
        // up to 4 vectors of K and 4 of V a lane in flight before their stores
        // (the copy is bound by the bytes in flight, not by instructions)
        for (int j0 = 0; j0 < per_tok; j0 += 128) {
            uint4 kv[4], vv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * 32 + lane;
                if (j < per_tok) {
                    kv[u] = __ldg(ks + j);
                    vv[u] = __ldg(vs + j);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = j0 + u * 32 + lane;
                if (j < per_tok) {
                    const int g = j >> log2hv, v = j & (hv - 1);
                    const int64_t dst = ((row0 + g) * p.page_size + slot) * hv + v;
                    p.k_pages[dst] = kv[u];
                    p.v_pages[dst] = vv[u];
                }
            }
        }
    }
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < p.batch; b += blockDim.x) {
            if (p.seq_lens[b] != p.old_len[b])
                atomicOr(p.err, SHKV_ERRF_SEQ_LEN);
            p.seq_lens[b] = p.old_len[b] + p.n_new;
        }
    }
}

cudaError_t launch_append(const AppendParams &p, int num_sms, cudaStream_t stream)
{
    const int64_t ntok = (int64_t)p.batch * p.n_new;
    int64_t blocks = (ntok + 7) / 8;                 // 8 warps a block, one token each
    if (blocks > (int64_t)num_sms * 8)
        blocks = (int64_t)num_sms * 8;
    if (blocks < 1)
        blocks = 1;
    return launch_pdl(shkv_append_kernel, (int)blocks, 256, 0u, stream, p);
}

// Log-sum-exp merge of split-KV partials.  One warp per (request, row); the
// lanes read the S log-sum-exps, agree on the max, then each lane reduces
// float4 slices of the S partial outputs with weights exp(lse_s - max).
__global__ void __launch_bounds__(256)
    shkv_merge_kernel(int n_splits, int batch, int rows, int head_dim, const float *__restrict__ o_part,
                      const float *__restrict__ lse_part, __nv_bfloat16 *__restrict__ out,
                      float *__restrict__ lse_out)
{
    pdl_wait_prior();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t nrow = (int64_t)batch * rows;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= nrow)
        return;
    float M = -INFINITY;
    for (int s = lane; s < n_splits; s += 32)
        M = fmaxf(M, lse_part[(int64_t)s * nrow + row]);
    for (int o = 16; o > 0; o >>= 1)
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float wsum = 0.f;
    if (M != -INFINITY)
        for (int s = lane; s < n_splits; s += 32)
            wsum += ex2_approx((lse_part[(int64_t)s * nrow + row] - M) * 1.4426950408889634f);
    for (int o = 16; o > 0; o >>= 1)
        wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int dq = head_dim / 4;
    for (int d4 = lane; d4 < dq; d4 += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            for (int s = 0; s < n_splits; ++s) {
                const float w = ex2_approx((lse_part[(int64_t)s * nrow + row] - M) * 1.4426950408889634f);
                if (w == 0.f)
                    continue;     // lse = -inf: an empty split, whose o is not read
                const float4 v = reinterpret_cast<const float4 *>(o_part + ((int64_t)s * nrow + row) * head_dim)[d4];
                acc.x += w * v.x;
                acc.y += w * v.y;
                acc.z += w * v.z;
                acc.w += w * v.w;
            }
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        uint2 packed;
        packed.x = *reinterpret_cast<uint32_t *>(&lo);
        packed.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(out + row * head_dim)[d4] = packed;
    }
    if (lane == 0 && lse_out)
        lse_out[row] = wsum > 0.f ? M + logf(wsum) : -INFINITY;
}

// One warp per request builds its row of the unit table: its shared pages
// then each decoder's tail pages, with each page's valid tokens and attending
// decoder.  The warp fits beside a decode CTA on an SM (at most 32 registers,
// no shared memory), so it runs while the previous kernel still does: it
// lets the next kernel be scheduled at once, reads the tables through L2
// only (they were written by work that completed before this kernel could
// start, see shkv_decode_attention_tails), writes tables at a position the
// previous decode does not read (else, wait_first, it waits at its start),
// and waits for the previous kernel at its end, so the decode after it starts
// only once both have completed.
__global__ void __maxnreg__(32) shkv_tails_unit_kernel(const __grid_constant__ TailsUnitParams p)
{
    if (p.wait_first)
        pdl_wait_prior();       // its table position may be in use by the previous decode
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int P = p.page_size;
    const int L = p.shared_len[b];
    const int S = (L + P - 1) / P;
    int U = S;
    for (int m = 0; m < p.n_models; ++m)
        U += (p.tail_len[b * p.n_models + m] + P - 1) / P;
    // three entries a lane per pass (four spill at 32 registers), their
    // table loads issued before any store
    constexpr int kUnroll = 3;
    for (int j0 = threadIdx.x; j0 < U; j0 += 32 * kUnroll) {
        int id[kUnroll];
        uint32_t info[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = j0 + 32 * u;
            id[u] = -1;
            info[u] = 0;
            if (j >= U)
                continue;
            if (j < S) {
                id[u] = __ldcg(p.block_table + (int64_t)b * p.bt_stride + j);
                info[u] = (uint32_t)(j == S - 1 ? L - j * P : P) | (kAllDecoders << 8);
            } else {
                int jt = j - S, m = 0;
                for (;; ++m) {
                    const int pages = (p.tail_len[b * p.n_models + m] + P - 1) / P;
                    if (jt < pages)
                        break;
                    jt -= pages;
                }
                const int T = p.tail_len[b * p.n_models + m];
                const int pages = (T + P - 1) / P;
                id[u] = __ldcg(p.tail_table + ((int64_t)b * p.n_models + m) * p.tt_stride + jt);
                info[u] = (uint32_t)(jt == pages - 1 ? T - jt * P : P) | ((uint32_t)m << 8);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = j0 + 32 * u;
            if (j < U) {
                p.unit_table[(int64_t)b * p.ustride + j] = id[u];
                p.unit_info[(int64_t)b * p.ustride + j] = info[u];
            }
        }
    }
    pdl_wait_prior();
}

cudaError_t launch_tails_units(const TailsUnitParams &p, cudaStream_t stream)
{
    return launch_pdl(shkv_tails_unit_kernel, p.batch, 32, 0u, stream, p);
}

cudaError_t launch_merge(int n_splits, int batch, int rows, int head_dim, const float *o_part,
                         const float *lse_part, __nv_bfloat16 *out, float *lse_out, cudaStream_t stream)
{
    const int64_t nrow = (int64_t)batch * rows;
    const int64_t blocks = (nrow + 7) / 8;
    if (blocks <= 0)
        return cudaSuccess;
    return launch_pdl(shkv_merge_kernel, (int)blocks, 256, 0u, stream, n_splits, batch, rows, head_dim, o_part,
                      lse_part, out, lse_out);
}

}  // namespace shkv
